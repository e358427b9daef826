// ddl_head.cu -- the token step around the layer stack ("把基础打牢" primer,
// §1.2 decode step: the last token's embedding row before the layers, and
// after them a token drawn from the logits of the last hidden state against
// the embedding table; Unsloth/Qwen-27B article §三: a vocabulary
// of about 152 thousand entries whose logits are produced chunk by chunk).
//
//  - embed_kernel: the rows of the bf16 embedding table for B token ids.
//  - head_prep_kernel: per sequence, the optional final RMSNorm factor and
//    the activation as m16n8k16 B fragments (fp16 hi/lo for INT4 weights,
//    bf16 hi/lo for bf16 weights, scaled by 2^-e so the largest |x w| lies in
//    [2^11, 2^12)).
//  - head_gemv_kernel: the vocabulary's 16-row tiles spread over the warps of
//    the grid; each warp streams a tile's packed blocks (codes expanded to
//    exact fp16 q and 16 q, warp-level tensor-core MMAs), writes the tile's
//    logits when asked, and folds the tile into a running (max, id of the
//    max, sum of exp(l - max)) per sequence: the vocabulary is reduced in
//    chunks and never held as a probability distribution.
//  - head_select_kernel: per sequence, the warps' records merged in a fixed
//    order (greedy id, log-sum-exp), and for top-k sampling a radix select of
//    the k-th largest logit, the k candidates in (logit descending, id
//    ascending) order and the inverse-CDF draw with the caller's uniform u.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <mutex>

#include "ddl_device.cuh"
#include "ddl_internal.h"

namespace ddl {
namespace {

constexpr int HEAD_THREADS = 256;  // 8 warps a CTA
constexpr int HEAD_CTAS_PER_SM = 2;
constexpr int SEL_THREADS = 1024;
constexpr int PREP_THREADS = 256;

int g_head_sms[64];
std::mutex g_head_mu;

int head_sms(int& sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= 64) return DDL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_head_mu);
  if (!g_head_sms[dev]) {
    int n = 0;
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_status(e);
    g_head_sms[dev] = n;
  }
  sms = g_head_sms[dev];
  return DDL_OK;
}

// n-tiles of 8 columns: two columns (hi, lo) per sequence, a power of two.
int head_ntn(int B) {
  int n = 1;
  while (4 * n < B) n *= 2;
  return n;
}

struct HeadLayout {
  int64_t xf, osc, rec, logits, total;
  int32_t ctas, nwarps;
};

int head_layout(int32_t D, int64_t V, int32_t B, HeadLayout& h) {
  int sms = 0;
  const int st = head_sms(sms);
  if (st) return st;
  h.ctas = sms * HEAD_CTAS_PER_SM;
  h.nwarps = h.ctas * (HEAD_THREADS / 32);
  int64_t off = 0;
  h.xf = off;
  off = align256(off + (int64_t)(D / 64) * 4 * head_ntn(B) * 32 * 8);
  h.osc = off;
  off = align256(off + (int64_t)DDL_MAX_BATCH * 4);
  h.rec = off;
  off = align256(off + (int64_t)B * h.nwarps * 16);
  h.logits = off;
  off = align256(off + (int64_t)B * V * 4);
  h.total = off;
  return DDL_OK;
}

// ------------------------------------------------------------------ packing
// Block (tile T, group grp) of a [V][D] matrix at (T * G + grp) * block bytes:
// the layers' block format (lane (g, t) of the INT4 codes holds rows g, g+8 at
// k = 16 j + 2t (+1, +8, +9) for the four k-slices j, then 16 bf16 scales as 8
// words (row g low, row g + 8 high); a bf16 block holds the four MMAs' A
// fragments).  Rows at or past V (the last tile's ragged end) are zero.
__device__ __forceinline__ uint32_t head_nib(const uint8_t* q, int64_t V, int D, int64_t row, int k) {
  if (row >= V) return 0u;
  const uint8_t byte = q[row * (D / 2) + k / 2];
  return (k & 1) ? (byte >> 4) : (byte & 0xFu);
}

__global__ void pack_head_int4_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s, int64_t V,
                                      int D, int64_t nblk, uint8_t* __restrict__ out) {
  const int G = D / 64;
  const int64_t per = nblk * 136;  // 128 code words + 8 scale words a block
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < per; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / 136;
    const int w = (int)(i % 136);
    const int64_t T = b / G;
    const int grp = (int)(b % G);
    uint32_t* ob = reinterpret_cast<uint32_t*>(out + b * QBLK_BYTES);
    if (w < 128) {
      const int lane = w / 4, j = w % 4, g = lane / 4, t = lane % 4;
      const int64_t rg = 16 * T + g, rh = rg + 8;
      const int k0 = grp * 64 + 16 * j + 2 * t;
      uint32_t wd = 0;
      wd |= head_nib(q, V, D, rg, k0) << 0;
      wd |= head_nib(q, V, D, rh, k0) << 4;
      wd |= head_nib(q, V, D, rg, k0 + 8) << 8;
      wd |= head_nib(q, V, D, rh, k0 + 8) << 12;
      wd |= head_nib(q, V, D, rg, k0 + 1) << 16;
      wd |= head_nib(q, V, D, rh, k0 + 1) << 20;
      wd |= head_nib(q, V, D, rg, k0 + 9) << 24;
      wd |= head_nib(q, V, D, rh, k0 + 9) << 28;
      ob[lane * 4 + j] = wd;
    } else {
      const int g = w - 128;
      const int64_t rg = 16 * T + g, rh = rg + 8;
      const uint32_t lo = rg < V ? s[rg * G + grp] : 0u, hi = rh < V ? s[rh * G + grp] : 0u;
      ob[128 + g] = lo | (hi << 16);
    }
  }
}

__global__ void pack_head_bf16_kernel(const uint16_t* __restrict__ w, int64_t V, int D, int64_t nblk,
                                      uint32_t* __restrict__ out) {
  const int G = D / 64;
  const int64_t nw = nblk * 512;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nw; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / 512;
    const int j = (int)(i % 512) / 128, lane = (int)(i % 128) / 4, reg = (int)(i % 4);
    const int g = lane / 4, t = lane % 4;
    const int64_t T = b / G;
    const int grp = (int)(b % G);
    const int64_t row = 16 * T + g + ((reg & 1) ? 8 : 0);
    const int k = grp * 64 + 16 * j + 2 * t + ((reg & 2) ? 8 : 0);
    out[i] = row < V ? *reinterpret_cast<const uint32_t*>(w + row * D + k) : 0u;
  }
}

// ------------------------------------------------------------------ embedding
__global__ void embed_kernel(const uint16_t* __restrict__ table, int64_t V, int D, const int32_t* __restrict__ tokens,
                             uint16_t* __restrict__ out, int32_t* __restrict__ bad) {
  const int b = blockIdx.x;
  const int32_t id = tokens[b];
  const bool ok = id >= 0 && (int64_t)id < V;
  if (!ok && threadIdx.x == 0 && bad) atomicOr(bad, 1);
  const uint4* src = reinterpret_cast<const uint4*>(table + (ok ? (int64_t)id : 0) * D);
  uint4* dst = reinterpret_cast<uint4*>(out + (int64_t)b * D);
  for (int i = threadIdx.x; i < D / 8; i += blockDim.x) dst[i] = ok ? src[i] : make_uint4(0u, 0u, 0u, 0u);
}

// ------------------------------------------------------------------ activation
// Fragment image: uint2 at ((grp * 4 + j) * NTN + n) * 32 + lane for k-slice j
// of group grp, n-tile n, lane (g, t): column g of n-tile n is sequence
// 4 n + g / 2, high part for even g, remainder for odd g; word 0 holds k
// = 16 j + 2t, +1 and word 1 k + 8, + 9 of the group.  Columns of sequences
// >= B are never written: they only reach accumulator columns nobody reads.
template <int WT>
__global__ void __launch_bounds__(PREP_THREADS) head_prep_kernel(const float* __restrict__ x,
                                                                 const uint16_t* __restrict__ nw, float eps, int D,
                                                                 int ntn, uint2* __restrict__ xf,
                                                                 float* __restrict__ osc) {
  __shared__ float red[2][PREP_THREADS / 32];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();  // the logits kernel may be scheduled (it waits for this one before reading x's fragments)
  const float* xb = x + (int64_t)b * D;
  float ss = 0.f, mx = 0.f;
  for (int k = tid; k < D; k += PREP_THREADS) {
    const float v = xb[k];
    const float w = nw ? bf16_bits_to_f32(nw[k]) : 1.f;
    ss = fmaf(v, v, ss);
    mx = fmaxf(mx, fabsf(v * w));
  }
  for (int o = 16; o; o >>= 1) {
    ss += __shfl_xor_sync(FULL, ss, o);
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
  }
  if (lane == 0) {
    red[0][warp] = ss;
    red[1][warp] = mx;
  }
  __syncthreads();
  ss = 0.f;
  mx = 0.f;
  for (int w = 0; w < PREP_THREADS / 32; ++w) {  // fixed order: the same sums every call
    ss += red[0][w];
    mx = fmaxf(mx, red[1][w]);
  }
  const int e = mx > 0.f ? ilogbf(mx) - 11 : 0;
  const float sdn = ldexpf(1.f, -e);
  const float r = nw ? 1.f / sqrtf(ss / (float)D + eps) : 1.f;
  if (tid == 0) osc[b] = ldexpf(1.f, e) * r;
  const int n = b >> 2, c = 2 * (b & 3);
  for (int i = tid; i < (D / 16) * 4; i += PREP_THREADS) {
    const int s = i >> 2, t = i & 3;
    const int k0 = 16 * s + 2 * t;
    float v[4];
    const int ks[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = xb[ks[q]] * (nw ? bf16_bits_to_f32(nw[ks[q]]) : 1.f) * sdn;
    uint32_t hw[2], lw[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const float2 pv = make_float2(v[2 * p], v[2 * p + 1]);
      if (WT == DDL_W_INT4) {
        const __half2 hh = __float22half2_rn(pv);
        const float2 hf = __half22float2(hh);
        const __half2 ll = __float22half2_rn(make_float2(pv.x - hf.x, pv.y - hf.y));
        hw[p] = *reinterpret_cast<const uint32_t*>(&hh);
        lw[p] = *reinterpret_cast<const uint32_t*>(&ll);
      } else {
        const __nv_bfloat162 hh = __float22bfloat162_rn(pv);
        const float2 hf = __bfloat1622float2(hh);
        const __nv_bfloat162 ll = __float22bfloat162_rn(make_float2(pv.x - hf.x, pv.y - hf.y));
        hw[p] = *reinterpret_cast<const uint32_t*>(&hh);
        lw[p] = *reinterpret_cast<const uint32_t*>(&ll);
      }
    }
    const int grp = s >> 2, j = s & 3;
    uint2* base = xf + ((int64_t)(grp * 4 + j) * ntn + n) * 32;
    base[4 * c + t] = make_uint2(hw[0], hw[1]);
    base[4 * (c + 1) + t] = make_uint2(lw[0], lw[1]);
  }
}

// ------------------------------------------------------------------ logits
struct HeadArgs {
  const uint8_t* w;    // packed head
  const uint2* xf;     // fragment image
  const float* osc;    // [B] 2^e * RMSNorm factor
  float* logits;       // [B][V] or nullptr
  float4* rec;         // [B][nwarps]: (max, id bits, sum of exp(l - max), 0)
  int64_t V;
  int32_t G, NTt, B, nwarps;
};

__device__ __forceinline__ uint4 ldg_stream128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_stream32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// (m, id, s) <- (m, id, s) merged with (m2, id2, s2); equal maxima keep the lower id.
__device__ __forceinline__ void lse_merge(float& m, int& id, float& s, float m2, int id2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    id = id2;
    s = s2;
    return;
  }
  const float nm = fmaxf(m, m2);
  s = s * expf(m - nm) + s2 * expf(m2 - nm);
  if (m2 > m || (m2 == m && id2 < id)) id = id2;
  m = nm;
}

// NTN n-tiles of 8 columns (4 sequences each); PER blocks of a tile per batch
// as independent MMA chains.
template <int WT, int NTN, int PER>
__global__ void __launch_bounds__(HEAD_THREADS, NTN <= 4 ? HEAD_CTAS_PER_SM : 1)
    head_gemv_kernel(const HeadArgs A) {
  pdl_trigger();
  pdl_wait();  // the activation fragments from the preparation kernel
  constexpr int BLK = WT == DDL_W_INT4 ? QBLK_BYTES : BF16_BLK_BYTES;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int gw = blockIdx.x * (HEAD_THREADS / 32) + (threadIdx.x >> 5);
  float osc[NTN], rm[NTN], rs[NTN];
  int ri[NTN];
#pragma unroll
  for (int n = 0; n < NTN; ++n) {
    const int b = 4 * n + t;
    osc[n] = b < A.B ? A.osc[b] : 0.f;
    rm[n] = -INFINITY;
    rs[n] = 0.f;
    ri[n] = 0x7fffffff;
  }
  const uint2* xl = A.xf + lane;
  const int G = A.G;
  for (int T = gw; T < A.NTt; T += A.nwarps) {
    float acc[NTN][2];
#pragma unroll
    for (int n = 0; n < NTN; ++n) acc[n][0] = acc[n][1] = 0.f;
    const uint8_t* tb = A.w + (int64_t)T * G * BLK;
#pragma unroll 1
    for (int g0 = 0; g0 < G; g0 += PER) {
      float c[PER][NTN][4];
#pragma unroll
      for (int i = 0; i < PER; ++i)
#pragma unroll
        for (int n = 0; n < NTN; ++n) c[i][n][0] = c[i][n][1] = c[i][n][2] = c[i][n][3] = 0.f;
      if (WT == DDL_W_INT4) {
        uint4 q[PER];
        uint32_t sw[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const bool in = g0 + i < G;  // past the tile's end: zero codes and scales
          const uint8_t* blk = tb + (int64_t)(in ? g0 + i : 0) * BLK;
          q[i] = in ? ldg_stream128(blk + lane * 16) : make_uint4(0u, 0u, 0u, 0u);
          sw[i] = in ? ldg_stream32(blk + BLK_BYTES + g * 4) : 0u;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int i = 0; i < PER; ++i) {
            const uint32_t w = j == 0 ? q[i].x : j == 1 ? q[i].y : j == 2 ? q[i].z : q[i].w;
            const uint32_t w8 = w >> 8;
            // 1024 + (q + 8) - 1032 = q and 1024 + 16 (q + 8) - 1152 = 16 q, exact in fp16
            const uint32_t a0 = hsub2_bits(lop3_merge(w, 0x000F000Fu, 0x64086408u), 0x64086408u);
            const uint32_t a1 = hsub2_bits(lop3_merge(w, 0x00F000F0u, 0x64806480u), 0x64806480u);
            const uint32_t a2 = hsub2_bits(lop3_merge(w8, 0x000F000Fu, 0x64086408u), 0x64086408u);
            const uint32_t a3 = hsub2_bits(lop3_merge(w8, 0x00F000F0u, 0x64806480u), 0x64806480u);
            const int gi = g0 + i < G ? g0 + i : G - 1;
#pragma unroll
            for (int n = 0; n < NTN; ++n) {
              const uint2 xv = __ldg(xl + ((int64_t)(gi * 4 + j) * NTN + n) * 32);
              mma_f16(c[i][n], a0, a1, a2, a3, xv.x, xv.y);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const float sg = bf16lo_f32(sw[i]), sh = bf16hi_f32(sw[i]) * 0.0625f;
#pragma unroll
          for (int n = 0; n < NTN; ++n) {
            acc[n][0] = fmaf(sg, c[i][n][0] + c[i][n][1], acc[n][0]);
            acc[n][1] = fmaf(sh, c[i][n][2] + c[i][n][3], acc[n][1]);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const bool in = g0 + i < G;
          const uint8_t* blk = tb + (int64_t)(in ? g0 + i : 0) * BLK;
          const int gi = in ? g0 + i : G - 1;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 a = in ? ldg_stream128(blk + j * 512 + lane * 16) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int n = 0; n < NTN; ++n) {
              const uint2 xv = __ldg(xl + ((int64_t)(gi * 4 + j) * NTN + n) * 32);
              mma_bf16(c[i][n], a.x, a.y, a.z, a.w, xv.x, xv.y);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < PER; ++i)
#pragma unroll
          for (int n = 0; n < NTN; ++n) {
            acc[n][0] += c[i][n][0] + c[i][n][1];
            acc[n][1] += c[i][n][2] + c[i][n][3];
          }
      }
    }
    // the tile's 16 logits per sequence: rows 16 T + g and + 8 of sequence 4 n + t
    const int64_t r0 = (int64_t)T * 16 + g, r1 = r0 + 8;
#pragma unroll
    for (int n = 0; n < NTN; ++n) {
      const int b = 4 * n + t;
      const bool sb = b < A.B;
      const float l0 = acc[n][0] * osc[n], l1 = acc[n][1] * osc[n];
      const bool v0 = sb && r0 < A.V, v1 = sb && r1 < A.V;
      if (A.logits) {
        if (v0) A.logits[(int64_t)b * A.V + r0] = l0;
        if (v1) A.logits[(int64_t)b * A.V + r1] = l1;
      }
      float m = v0 ? l0 : -INFINITY;
      int id = (int)r0;
      if (v1 && l1 > m) {
        m = l1;
        id = (int)r1;
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {  // lanes of the same t: the tile's 16 rows
        const float om = __shfl_xor_sync(FULL, m, o);
        const int oi = __shfl_xor_sync(FULL, id, o);
        if (om > m || (om == m && oi < id)) {
          m = om;
          id = oi;
        }
      }
      float s = 0.f;
      if (m != -INFINITY) s = (v0 ? expf(l0 - m) : 0.f) + (v1 ? expf(l1 - m) : 0.f);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) s += __shfl_xor_sync(FULL, s, o);
      lse_merge(rm[n], ri[n], rs[n], m, id, s);
    }
  }
#pragma unroll
  for (int n = 0; n < NTN; ++n) {
    const int b = 4 * n + t;
    if (b < A.B && g == 0)
      A.rec[(int64_t)b * A.nwarps + gw] = make_float4(rm[n], __int_as_float(ri[n]), rs[n], 0.f);
  }
}

// ------------------------------------------------------------------ selection
struct SelArgs {
  const float4* rec;
  const float* logits;  // [B][V] (top-k sampling only)
  const float* u;       // [B] (top-k sampling only)
  int32_t* token;
  float* lse;
  int64_t V;
  int32_t nwarps, top_k;
  float temperature;
};

// Order-preserving map of an fp32 value to an unsigned key.
__device__ __forceinline__ uint32_t fkey(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Exclusive prefix sum over the block (fixed order), returns the total.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* wsum, uint32_t& excl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(FULL, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < SEL_THREADS / 32 ? wsum[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, w, o);
      if (lane >= o) w += y;
    }
    if (lane < SEL_THREADS / 32) wsum[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t before = warp ? wsum[warp - 1] : 0u;
  excl = before + inc - v;
  const uint32_t total = wsum[SEL_THREADS / 32 - 1];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(SEL_THREADS) head_select_kernel(const SelArgs S) {
  __shared__ float rm_s[SEL_THREADS], rs_s[SEL_THREADS];
  __shared__ int ri_s[SEL_THREADS];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t wsum[SEL_THREADS / 32];
  __shared__ unsigned long long cand[DDL_MAX_TOP_K];
  __shared__ float cw[DDL_MAX_TOP_K];
  pdl_wait();  // the logits kernel's records and logits
  __shared__ uint32_t sh_digit, sh_krem;
  const int b = blockIdx.x, tid = threadIdx.x;
  // 1. the warps' records, merged in a fixed order: strided runs, then a tree
  float m = -INFINITY, s = 0.f;
  int id = 0x7fffffff;
  for (int i = tid; i < S.nwarps; i += SEL_THREADS) {
    const float4 r = S.rec[(int64_t)b * S.nwarps + i];
    lse_merge(m, id, s, r.x, __float_as_int(r.y), r.z);
  }
  rm_s[tid] = m;
  rs_s[tid] = s;
  ri_s[tid] = id;
  __syncthreads();
  for (int h = SEL_THREADS / 2; h > 0; h >>= 1) {
    if (tid < h) {
      float mm = rm_s[tid], ss = rs_s[tid];
      int ii = ri_s[tid];
      lse_merge(mm, ii, ss, rm_s[tid + h], ri_s[tid + h], rs_s[tid + h]);
      rm_s[tid] = mm;
      rs_s[tid] = ss;
      ri_s[tid] = ii;
    }
    __syncthreads();
  }
  if (tid == 0) {
    if (S.lse) S.lse[b] = rm_s[0] + logf(rs_s[0]);
    if (S.top_k <= 1) S.token[b] = ri_s[0];
  }
  if (S.top_k <= 1) return;
  // 2. top-k: the k-th largest key by radix select, most significant byte first
  const float* L = S.logits + (int64_t)b * S.V;
  const int k = (int64_t)S.top_k < S.V ? S.top_k : (int)S.V;
  uint32_t prefix = 0u, mask = 0u, krem = (uint32_t)k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += SEL_THREADS) hist[i] = 0u;
    __syncthreads();
    for (int64_t i = tid; i < S.V; i += SEL_THREADS) {
      const uint32_t key = fkey(L[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t cum = 0u;
      int d = 255;
      for (; d > 0; --d) {
        if (cum + hist[d] >= krem) break;
        cum += hist[d];
      }
      sh_digit = (uint32_t)d;
      sh_krem = krem - cum;
    }
    __syncthreads();
    prefix |= sh_digit << shift;
    mask |= 255u << shift;
    krem = sh_krem;
    __syncthreads();
  }
  const uint32_t tau = prefix;          // the k-th largest key
  const uint32_t n_gt = (uint32_t)k - krem;  // keys above tau; krem of the keys equal to tau are taken
  // 3. the candidates in id order: each thread a contiguous run of ids
  const int64_t per = (S.V + SEL_THREADS - 1) / SEL_THREADS;
  const int64_t i0 = (int64_t)tid * per, i1 = i0 + per < S.V ? i0 + per : S.V;
  uint32_t ngt = 0u, neq = 0u;
  for (int64_t i = i0; i < i1; ++i) {
    const uint32_t key = fkey(L[i]);
    ngt += key > tau;
    neq += key == tau;
  }
  uint32_t ogt, oeq;
  block_scan(ngt, wsum, ogt);
  block_scan(neq, wsum, oeq);
  for (int64_t i = i0; i < i1; ++i) {
    const uint32_t key = fkey(L[i]);
    const unsigned long long c = ((unsigned long long)key << 32) | (uint32_t)~(uint32_t)i;
    if (key > tau) {
      cand[ogt++] = c;
    } else if (key == tau) {
      if (oeq < krem) cand[n_gt + oeq] = c;
      ++oeq;
    }
  }
  int kp = 1;
  while (kp < k) kp <<= 1;
  for (int i = k + tid; i < kp; i += SEL_THREADS) cand[i] = 0ull;  // below every candidate
  __syncthreads();
  // 4. bitonic sort, descending: logit descending, then id ascending (~id descending)
  for (int size = 2; size <= kp; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < kp; i += SEL_THREADS) {
        const int p = i ^ stride;
        if (p > i) {
          const unsigned long long a = cand[i], c = cand[p];
          const bool desc = (i & size) == 0;
          if (desc ? (a < c) : (a > c)) {
            cand[i] = c;
            cand[p] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  // 5. weights exp((l - l_max) / T) and the inverse-CDF draw
  const float lmax = fkey_inv((uint32_t)(cand[0] >> 32));
  for (int i = tid; i < k; i += SEL_THREADS) cw[i] = expf((fkey_inv((uint32_t)(cand[i] >> 32)) - lmax) / S.temperature);
  __syncthreads();
  if (tid == 0) {
    float c = 0.f;
    for (int i = 0; i < k; ++i) {
      c += cw[i];
      cw[i] = c;
    }
    float u = S.u[b];
    u = u > 0.f ? u : 0.f;
    const float target = u * c;
    int j = 0;
    while (j < k - 1 && !(cw[j] > target)) ++j;
    S.token[b] = (int32_t)~(uint32_t)(cand[j] & 0xffffffffull);
  }
}

}  // namespace
}  // namespace ddl

using namespace ddl;

extern "C" size_t ddl_packed_head_bytes(int32_t D, int64_t V, ddl_wtype wtype) {
  if (D <= 0 || D % 64 || V <= 0 || V > 0x7fffffffLL) return 0;
  if (wtype != DDL_W_INT4 && wtype != DDL_W_BF16) return 0;
  const int64_t nblk = ((V + 15) / 16) * (D / 64);
  return (size_t)(nblk * (wtype == DDL_W_INT4 ? QBLK_BYTES : BF16_BLK_BYTES));
}

extern "C" int ddl_pack_head(const ddl_mat* w, int32_t D, int64_t V, ddl_wtype wtype, void* packed_out,
                             void* stream) {
  if (!w || !packed_out || D <= 0 || V <= 0) return DDL_ERR_ARG;
  if (D % 64 || V > 0x7fffffffLL) return DDL_ERR_SHAPE;
  if (wtype != DDL_W_INT4 && wtype != DDL_W_BF16) return DDL_ERR_UNSUPPORTED;
  if (!aligned16(packed_out)) return DDL_ERR_ALIGN;
  const int64_t nblk = ((V + 15) / 16) * (D / 64);
  cudaStream_t s = (cudaStream_t)stream;
  if (wtype == DDL_W_INT4) {
    if (!w->q || !w->scale) return DDL_ERR_ARG;
    const int64_t work = nblk * 136;
    const int blocks = (int)((work + 255) / 256 < 65535 * 16 ? (work + 255) / 256 : 65535 * 16);
    pack_head_int4_kernel<<<blocks, 256, 0, s>>>(w->q, w->scale, V, D, nblk, (uint8_t*)packed_out);
  } else {
    if (!w->w) return DDL_ERR_ARG;
    if ((uintptr_t)w->w & 3) return DDL_ERR_ALIGN;
    const int64_t work = nblk * 512;
    const int blocks = (int)((work + 255) / 256 < 65535 * 16 ? (work + 255) / 256 : 65535 * 16);
    pack_head_bf16_kernel<<<blocks, 256, 0, s>>>(w->w, V, D, nblk, (uint32_t*)packed_out);
  }
  return cuda_status(cudaGetLastError());
}

extern "C" int ddl_embed(const uint16_t* table, int64_t V, int32_t D, const int32_t* tokens, int32_t B,
                         uint16_t* x_out, int32_t* bad_out, void* stream) {
  if (!table || !tokens || !x_out || V <= 0 || D <= 0 || B <= 0) return DDL_ERR_ARG;
  if (D % 64) return DDL_ERR_SHAPE;
  if (B > DDL_MAX_BATCH) return DDL_ERR_UNSUPPORTED;
  if (!aligned16(table) || !aligned16(x_out) || ((uintptr_t)tokens & 3) || ((uintptr_t)bad_out & 3))
    return DDL_ERR_ALIGN;
  embed_kernel<<<B, 128, 0, (cudaStream_t)stream>>>(table, V, D, tokens, x_out, bad_out);
  return cuda_status(cudaGetLastError());
}

extern "C" size_t ddl_head_workspace_bytes(int32_t D, int64_t V, int32_t B) {
  if (D <= 0 || D % 64 || V <= 0 || V > 0x7fffffffLL || B < 1 || B > DDL_MAX_BATCH) return 0;
  HeadLayout h;
  if (head_layout(D, V, B, h)) return 0;
  return (size_t)h.total;
}

template <int WT, int NTN, int PER>
static cudaError_t launch_gemv(const HeadLayout& h, const HeadArgs& a, cudaStream_t s) {
  void* args[] = {const_cast<HeadArgs*>(&a)};
  return launch_pdl((const void*)head_gemv_kernel<WT, NTN, PER>, dim3(h.ctas), dim3(HEAD_THREADS), args, 0, s);
}

template <int WT>
static cudaError_t launch_gemv_ntn(int ntn, const HeadLayout& h, const HeadArgs& a, cudaStream_t s) {
  constexpr int P1 = WT == DDL_W_INT4 ? 8 : 2;
  switch (ntn) {
    case 1: return launch_gemv<WT, 1, P1>(h, a, s);
    case 2: return launch_gemv<WT, 2, P1 / 2>(h, a, s);
    case 4: return launch_gemv<WT, 4, (P1 / 4 > 0 ? P1 / 4 : 1)>(h, a, s);
    case 8: return launch_gemv<WT, 8, 1>(h, a, s);
    default: return launch_gemv<WT, 16, 1>(h, a, s);
  }
}

extern "C" int ddl_lm_head(int32_t D, int64_t V, ddl_wtype wtype, const void* head_packed, const uint16_t* norm_f,
                           float eps, int32_t B, const float* x, int32_t top_k, float temperature, const float* u,
                           int32_t* token_out, float* logits_out, float* lse_out, void* workspace, size_t ws_bytes,
                           void* stream) {
  if (!head_packed || !x || !token_out || !workspace || D <= 0 || V <= 0 || B <= 0 || top_k < 0) return DDL_ERR_ARG;
  if (D % 64 || V > 0x7fffffffLL) return DDL_ERR_SHAPE;
  if (wtype != DDL_W_INT4 && wtype != DDL_W_BF16) return DDL_ERR_UNSUPPORTED;
  if (B > DDL_MAX_BATCH || top_k > DDL_MAX_TOP_K) return DDL_ERR_UNSUPPORTED;
  if (!(eps >= 0.f)) return DDL_ERR_ARG;
  if (top_k > 1 && (!u || !(temperature > 0.f) || !(temperature < INFINITY))) return DDL_ERR_ARG;
  if (!aligned16(head_packed) || !aligned16(x) || !aligned16(workspace) || ((uintptr_t)token_out & 3) ||
      ((uintptr_t)logits_out & 3) || ((uintptr_t)lse_out & 3) || ((uintptr_t)u & 3) || ((uintptr_t)norm_f & 1))
    return DDL_ERR_ALIGN;
  HeadLayout h;
  int st = head_layout(D, V, B, h);
  if (st) return st;
  if ((int64_t)ws_bytes < h.total) return DDL_ERR_WORKSPACE;
  uint8_t* ws = (uint8_t*)workspace;
  cudaStream_t s = (cudaStream_t)stream;
  const int ntn = head_ntn(B);
  uint2* xf = reinterpret_cast<uint2*>(ws + h.xf);
  float* osc = reinterpret_cast<float*>(ws + h.osc);
  if (wtype == DDL_W_INT4)
    head_prep_kernel<DDL_W_INT4><<<B, PREP_THREADS, 0, s>>>(x, norm_f, eps, D, ntn, xf, osc);
  else
    head_prep_kernel<DDL_W_BF16><<<B, PREP_THREADS, 0, s>>>(x, norm_f, eps, D, ntn, xf, osc);
  if ((st = cuda_status(cudaGetLastError()))) return st;
  HeadArgs a;
  a.w = (const uint8_t*)head_packed;
  a.xf = xf;
  a.osc = osc;
  float* logits = logits_out ? logits_out : (top_k > 1 ? reinterpret_cast<float*>(ws + h.logits) : nullptr);
  a.logits = logits;
  a.rec = reinterpret_cast<float4*>(ws + h.rec);
  a.V = V;
  a.G = D / 64;
  a.NTt = (int32_t)((V + 15) / 16);
  a.B = B;
  a.nwarps = h.nwarps;
  const cudaError_t e = wtype == DDL_W_INT4 ? launch_gemv_ntn<DDL_W_INT4>(ntn, h, a, s)
                                            : launch_gemv_ntn<DDL_W_BF16>(ntn, h, a, s);
  if ((st = cuda_status(e))) return st;
  SelArgs sa;
  sa.rec = a.rec;
  sa.logits = logits;
  sa.u = u;
  sa.token = token_out;
  sa.lse = lse_out;
  sa.V = V;
  sa.nwarps = h.nwarps;
  sa.top_k = top_k;
  sa.temperature = temperature;
  void* sargs[] = {&sa};
  return cuda_status(launch_pdl((const void*)head_select_kernel, dim3(B), dim3(SEL_THREADS), sargs, 0, s));
}
