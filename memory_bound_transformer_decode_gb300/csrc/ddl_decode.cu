// ddl_decode.cu -- the decode step: one persistent kernel that streams every
// weight and KV byte of an L-layer stack once, and its host runtime.
//
// Per layer the kernel runs six stages (primer "把基础打牢" §1.1 block, §1.2
// decode_step):
//   QKV  : rmsnorm(x) folded into the GEMV (W (x*w1)) * r, INT4 codes expanded
//          in registers and multiplied on the tensor cores, RoPE on q and k,
//          bf16 k and v appended to the cache at slot pos (Unsloth/Qwen-27B
//          article §二.1 fused RMSNorm+RoPE, §二.3 in-register 4-bit expansion)
//   ATT  : split-KV GQA decode attention: each K/V head is read once, in
//          place, for its whole query group (same article §二.2), with an
//          online softmax per 16-key tile (FlashAttention-style tiling, roofline
//          reply §四)
//   COMB : merge of the split-KV partial softmax states
//   WO   : y = x + attn Wo
//   GU   : rmsnorm(y) folded into the gate/up GEMV, silu(g) * u in the epilogue
//          (Unsloth/Qwen-27B article §二.1 fused SwiGLU)
//   DOWN : z = y + a Wd
// Every warp owns a ring of DEPTH shared-memory slots filled by 1-D TMA bulk
// copies; its lane 0 keeps DEPTH slots in flight, running ahead across stage
// (and layer) boundaries because weights and the KV history do not depend on
// the token being decoded.  Stages are separated by a grid-wide barrier (one
// cooperative launch for the whole stack) or by kernel boundaries (one launch
// per stage).  All waits are bounded: a wait that gives up sets the status
// word in the workspace and the kernel returns.
#include <math.h>
#include <mutex>
#include <stdio.h>
#include <string.h>

#include "ddl_device.cuh"
#include "ddl_internal.h"

namespace ddl {

// ------------------------------------------------------------------ shared memory
constexpr int SM_RING = 0;
constexpr int SM_RING_BYTES = NW * DEPTH * SLOT_BYTES;
constexpr int SM_BARS = SM_RING_BYTES;
constexpr int SM_SCR = SM_BARS + 256;
constexpr int XF_BYTES = 2 * GC * 4 * (2 * MAX_B) * 4 * 8;  // x fragments, 2 k-chunks
constexpr int SX_BYTES = 2 * GC * MAX_B * 4;                // per-group sums of x
constexpr int SM_SCR_BYTES = 70 * 1024;
constexpr int SM_MISC = SM_SCR + SM_SCR_BYTES;
constexpr int SM_MISC_BYTES = 2048;
constexpr int SM_TOTAL = SM_MISC + SM_MISC_BYTES;
static_assert(XF_BYTES + SX_BYTES <= SM_SCR_BYTES, "x fragments do not fit");
static_assert(NW * 2 * MAX_GH * (128 + 2) * 4 <= SM_SCR_BYTES, "attention records do not fit");
static_assert(SM_TOTAL <= 227 * 1024, "shared memory budget");

struct Misc {
  float rnorm[MAX_B];
  float escale[2][MAX_B];  // 2^e of each staged k-chunk and sequence
  float edown[2][MAX_B];   // 2^-e
  float red[NW][3 * MAX_B];
  float rope[64][2];       // cos, sin of pair i at position pos
  int kc_lo, nkc;
  int abort;
  int seg_n[NW];
  long long seg_first[NW], seg_last[NW];
};
static_assert(sizeof(Misc) <= SM_MISC_BYTES, "misc");

enum SlotKind { SK_GEMV = 0, SK_K = 1, SK_V = 2 };

struct SlotDesc {
  int kind, layer, mk, cnt;
  int64_t a;
};
struct Cursor {
  int s;
  int64_t pos, end;
};
struct Ring {
  uint32_t slot0, bar0, n_issued, n_done;
  __device__ __forceinline__ uint32_t slot(uint32_t n) const { return slot0 + (n % DEPTH) * SLOT_BYTES; }
  __device__ __forceinline__ uint32_t bar(uint32_t n) const { return bar0 + (n % DEPTH) * 8; }
  __device__ __forceinline__ uint32_t parity(uint32_t n) const { return (n / DEPTH) & 1; }
};

// ------------------------------------------------------------------ work split
__device__ __forceinline__ void att_range(const Params& P, int64_t& lo, int64_t& hi) {
  const int64_t Ta = (int64_t)P.B * P.Hkv * P.nt_att, C = gridDim.x;
  const int64_t clo = range_lo(Ta, C, blockIdx.x), chi = range_lo(Ta, C, blockIdx.x + 1);
  const int w = threadIdx.x >> 5;
  lo = clo + range_lo(chi - clo, NW, w);
  hi = clo + range_lo(chi - clo, NW, w + 1);
}
__device__ __forceinline__ int slot_blocks(const Params& P) {
  return P.wtype == DDL_W_INT4 ? BLKS_PER_SLOT : BF16_BLKS_PER_SLOT;
}
__device__ __forceinline__ void cursor_range(const Params& P, int s, int64_t wg, int64_t W,
                                             int64_t& lo, int64_t& hi) {
  const int st = s % NSTAGE;
  if (st == ST_ATT) {
    att_range(P, lo, hi);
    lo *= 2;
    hi *= 2;
  } else if (st == ST_COMB) {
    lo = hi = 0;
  } else {
    const int64_t T = P.mg[stage_mat(st)].T;
    lo = range_lo(T, W, wg);
    hi = range_lo(T, W, wg + 1);
  }
}
__device__ __forceinline__ bool cursor_next(const Params& P, Cursor& c, int64_t wg, int64_t W,
                                            SlotDesc& d) {
  while (c.pos >= c.end) {
    if (++c.s >= P.stage_end) return false;
    cursor_range(P, c.s, wg, W, c.pos, c.end);
  }
  const int st = c.s % NSTAGE;
  d.layer = c.s / NSTAGE;
  if (st == ST_ATT) {
    const int64_t tile = c.pos >> 1;
    d.kind = (c.pos & 1) ? SK_V : SK_K;
    d.a = tile;
    const int64_t i = tile % P.nt_att;
    const int64_t rows = P.pos - 16 * i;
    d.cnt = (int)(rows < 0 ? 0 : rows > 16 ? 16 : rows);
    d.mk = -1;
    c.pos += 1;
  } else {
    d.kind = SK_GEMV;
    d.mk = stage_mat(st);
    d.a = c.pos;
    const int64_t left = c.end - c.pos;
    d.cnt = (int)(left < slot_blocks(P) ? left : slot_blocks(P));
    c.pos += d.cnt;
  }
  return true;
}

template <int HD>
__device__ __forceinline__ void issue_slot(const Params& P, const SlotDesc& d, uint32_t slot,
                                           uint32_t bar, int lane, uint64_t policy) {
  constexpr int ROWB = HD * 2 + 16;
  const LayerDev& Ld = P.layers[d.layer];
  if (d.kind == SK_GEMV) {
    if (lane == 0) {
      const MatGeom& m = P.mg[d.mk];
      const bool q4 = P.wtype == DDL_W_INT4;
      const uint32_t wb = d.cnt * (q4 ? BLK_BYTES : BF16_BLK_BYTES);
      const uint32_t sb = q4 ? d.cnt * SCL_BYTES : 0;
      mbar_arrive_expect_tx(bar, wb + sb);
      bulk_g2s_evict_first(slot, Ld.packed + m.woff + d.a * (q4 ? BLK_BYTES : BF16_BLK_BYTES), wb,
                           bar, policy);
      if (sb) bulk_g2s_evict_first(slot + BLKS_PER_SLOT * BLK_BYTES, Ld.packed + m.soff + d.a * SCL_BYTES,
                                   sb, bar, policy);
    }
  } else {
    const int64_t seq = d.a / P.nt_att, i = d.a % P.nt_att;
    const uint16_t* base = (d.kind == SK_K ? Ld.kc : Ld.vc) + (seq * P.s_max + 16 * i) * HD;
    if (lane == 0) mbar_arrive_expect_tx(bar, d.cnt * HD * 2);
    if (lane < d.cnt) bulk_g2s_evict_first(slot + lane * ROWB, base + lane * HD, HD * 2, bar, policy);
  }
}

// Release the slot just consumed and refill the ring from the cursor.
template <int HD>
__device__ __forceinline__ void ring_advance(const Params& P, Ring& R, Cursor& prod, int64_t wg,
                                             int64_t W, int lane, uint64_t policy) {
  __syncwarp();
  SlotDesc d;
  if (cursor_next(P, prod, wg, W, d)) {
    fence_proxy_async_smem();  // every issuing lane: earlier generic smem accesses first
    issue_slot<HD>(P, d, R.slot(R.n_issued), R.bar(R.n_issued), lane, policy);
    R.n_issued++;
  }
  R.n_done++;
}

// ------------------------------------------------------------------ block-wide reduce
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}

// Layer input x (fp32 residual) of global layer gl, element i of sequence b.
__device__ __forceinline__ float layer_input(const Params& P, int gl, int b, int i) {
  const int64_t o = (int64_t)b * P.D + i;
  if (gl == 0) return P.resid_in ? __ldcg(P.resid_in + o) : bf16_bits_to_f32(P.x_bf16[o]);
  return __ldcg(P.Z + (int64_t)((gl - 1) & 1) * P.B * P.D + o);
}

// ------------------------------------------------------------------ GEMV prologue
// Stages this CTA's share of the activation as m16n8k16 B fragments: column
// 2b is the fp16 "high" part of sequence b's x (times the norm weight and
// 2^-e), column 2b+1 the fp16 remainder, so x is carried to ~22 bits.  Also
// computes the RMSNorm factor r (QKV, GU), the per-k-chunk power-of-two scale
// and, for INT4, the per-group sums of x used to remove the +8 code offset.
template <int HD, int WT>
__device__ void gemv_prologue(const Params& P, int layer, int st, const MatGeom& m, int64_t W,
                              uint8_t* smem, Misc& M) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, B2 = 2 * B, gl = P.l0 + layer;
  const LayerDev& Ld = P.layers[layer];
  const int64_t clo = range_lo(m.T, W, (int64_t)blockIdx.x * NW);
  const int64_t chi = range_lo(m.T, W, (int64_t)(blockIdx.x + 1) * NW);
  int kc_lo = 0, nkc = 0;
  if (clo < chi) {
    int a, b_, kc_hi;
    block_coord(m, clo, kc_lo, a, b_);
    block_coord(m, chi - 1, kc_hi, a, b_);
    nkc = kc_hi - kc_lo + 1;
  }
  const float* xf32 = nullptr;
  const uint16_t* nw = nullptr;
  bool from_input = false;
  switch (st) {
    case ST_QKV: from_input = true; nw = Ld.norm1; break;
    case ST_WO: xf32 = P.attn; break;
    case ST_GU: xf32 = P.y; nw = Ld.norm2; break;
    default: xf32 = P.a; break;
  }
  const int K = m.K;
  const int k_lo = kc_lo * GC * DDL_GROUP;
  const int k_hi = min(K, (kc_lo + nkc) * GC * DDL_GROUP);
  auto load = [&](int b, int k) -> float {
    return from_input ? layer_input(P, gl, b, k) : __ldcg(xf32 + (int64_t)b * K + k);
  };
  if (st == ST_QKV && tid < HD / 2) {
    const double theta = pow(P.rope_base, -2.0 * (double)tid / (double)HD);
    double sn, cs;
    sincos((double)P.pos * theta, &sn, &cs);
    M.rope[tid][0] = (float)cs;
    M.rope[tid][1] = (float)sn;
  }
  // pass 1: sum of squares (norm stages, whole vector) and max |x'| per staged chunk
  for (int b = 0; b < B; ++b) {
    float ss = 0.f, mx0 = 0.f, mx1 = 0.f;
    const int a0 = nw ? 0 : k_lo, a1 = nw ? K : k_hi;
    for (int k = a0 + tid; k < a1; k += NTHREADS) {
      const float x = load(b, k);
      ss = fmaf(x, x, ss);
      if (k >= k_lo && k < k_hi) {
        const float v = fabsf(nw ? x * bf16_bits_to_f32(nw[k]) : x);
        if (k - k_lo < GC * DDL_GROUP) mx0 = fmaxf(mx0, v);
        else mx1 = fmaxf(mx1, v);
      }
    }
    ss = warp_sum(ss);
    mx0 = warp_max(mx0);
    mx1 = warp_max(mx1);
    if (lane == 0) {
      M.red[warp][3 * b + 0] = ss;
      M.red[warp][3 * b + 1] = mx0;
      M.red[warp][3 * b + 2] = mx1;
    }
  }
  __syncthreads();
  if (tid < B) {
    float ss = 0.f, mx0 = 0.f, mx1 = 0.f;
    for (int w = 0; w < NW; ++w) {
      ss += M.red[w][3 * tid + 0];
      mx0 = fmaxf(mx0, M.red[w][3 * tid + 1]);
      mx1 = fmaxf(mx1, M.red[w][3 * tid + 2]);
    }
    M.rnorm[tid] = nw ? 1.0f / sqrtf(ss / (float)K + P.eps) : 1.0f;
    const float mxs[2] = {mx0, mx1};
    for (int c = 0; c < 2; ++c) {
      const int e = mxs[c] > 0.f ? ilogbf(mxs[c]) - 11 : 0;
      M.escale[c][tid] = ldexpf(1.0f, e);
      M.edown[c][tid] = ldexpf(1.0f, -e);
    }
  }
  if (tid == 0) {
    M.kc_lo = kc_lo;
    M.nkc = nkc;
  }
  __syncthreads();
  // pass 2: fragments.  Item = (chunk, group, sequence, j, t); 16 consecutive
  // threads cover one (chunk, group, sequence).
  uint2* xf = reinterpret_cast<uint2*>(smem + SM_SCR);
  float* Sx = reinterpret_cast<float*>(smem + SM_SCR + XF_BYTES);
  const int n_items = nkc * GC * B * 16;
  for (int it0 = 0; it0 < n_items; it0 += NTHREADS) {
    const int it = it0 + tid;
    const int jt = it & 15, j = jt >> 2, t = jt & 3;
    int rest = it >> 4;
    const int b = rest % B;
    rest /= B;
    const int gi = rest % GC, kcl = rest / GC;
    const bool valid = it < n_items && gi < chunk_groups(m, kc_lo + kcl);
    double part = 0.0;
    if (valid) {
      const int k0 = (kc_lo + kcl) * GC * DDL_GROUP + gi * DDL_GROUP + 16 * j + 2 * t;
      const int kk[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
      float hi[4], lo[4];
      const float sc = M.edown[kcl][b];
      for (int e = 0; e < 4; ++e) {
        float x = load(b, kk[e]);
        if (nw) x *= bf16_bits_to_f32(nw[kk[e]]);
        x *= sc;
        if (WT == DDL_W_INT4) {
          hi[e] = __half2float(__float2half_rn(x));
          lo[e] = __half2float(__float2half_rn(x - hi[e]));
        } else {
          hi[e] = __bfloat162float(__float2bfloat16_rn(x));
          lo[e] = __bfloat162float(__float2bfloat16_rn(x - hi[e]));
        }
        part += (double)hi[e] + (double)lo[e];
      }
      const int base = (((kcl * GC + gi) * 4 + j) * B2) * 4 + t;
      if (WT == DDL_W_INT4) {
        xf[base + (2 * b) * 4] = make_uint2(pack_f16x2(hi[0], hi[1]), pack_f16x2(hi[2], hi[3]));
        xf[base + (2 * b + 1) * 4] = make_uint2(pack_f16x2(lo[0], lo[1]), pack_f16x2(lo[2], lo[3]));
      } else {
        xf[base + (2 * b) * 4] = make_uint2(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]));
        xf[base + (2 * b + 1) * 4] =
            make_uint2(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]));
      }
    }
    for (int o = 8; o; o >>= 1) part += __shfl_xor_sync(FULL, part, o);
    if (valid && jt == 0) Sx[(kcl * GC + gi) * MAX_B + b] = (float)part;
  }
  __syncthreads();
}

// ------------------------------------------------------------------ GEMV epilogues
// Lane (g, t) holds rows g and g+8 of tile T for sequence t.
template <int HD>
__device__ void gemv_epilogue(const Params& P, int layer, int st, int T, float v0, float v1,
                              const Misc& M) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  if (t >= P.B) return;
  const int gl = P.l0 + layer;
  const LayerDev& Ld = P.layers[layer];
  if (st == ST_QKV) {
    const float r = M.rnorm[t];
    v0 *= r;
    v1 *= r;
    const int tph = HD / 16, head = T / tph, i = 8 * (T % tph) + g;
    if (head < P.Hq + P.Hkv) {  // RoPE on q and k: pair (i, i + hd/2)
      const float c = M.rope[i][0], s = M.rope[i][1], a = v0, b = v1;
      v0 = a * c - b * s;
      v1 = a * s + b * c;
    }
    if (head < P.Hq) {
      float* qp = P.q + (int64_t)t * P.Hq * HD + (int64_t)head * HD;
      qp[i] = v0;
      qp[i + HD / 2] = v1;
    } else {
      const bool is_k = head < P.Hq + P.Hkv;
      const int kvh = is_k ? head - P.Hq : head - P.Hq - P.Hkv;
      uint16_t* row = (is_k ? Ld.kc : Ld.vc) + (((int64_t)t * P.Hkv + kvh) * P.s_max + P.pos) * HD;
      row[i] = f32_to_bf16_bits(v0);
      row[i + HD / 2] = f32_to_bf16_bits(v1);
    }
  } else if (st == ST_WO) {
    const int r0 = 16 * T + g, r1 = r0 + 8;
    float* y = P.y + (int64_t)t * P.D;
    y[r0] = layer_input(P, gl, t, r0) + v0;
    y[r1] = layer_input(P, gl, t, r1) + v1;
  } else if (st == ST_GU) {
    const float r = M.rnorm[t], gt = v0 * r, up = v1 * r;
    P.a[(int64_t)t * P.dff + 8 * T + g] = gt / (1.0f + expf(-gt)) * up;
  } else {
    const int r0 = 16 * T + g, r1 = r0 + 8;
    const float* y = P.y + (int64_t)t * P.D;
    const float z0 = __ldcg(y + r0) + v0, z1 = __ldcg(y + r1) + v1;
    float* Z = P.Z + (int64_t)(gl & 1) * P.B * P.D + (int64_t)t * P.D;
    Z[r0] = z0;
    Z[r1] = z1;
    if (P.final_last && layer == P.L - 1) {
      if (P.resid_out) {
        P.resid_out[(int64_t)t * P.D + r0] = z0;
        P.resid_out[(int64_t)t * P.D + r1] = z1;
      }
      if (P.out_bf16) {
        P.out_bf16[(int64_t)t * P.D + r0] = f32_to_bf16_bits(z0);
        P.out_bf16[(int64_t)t * P.D + r1] = f32_to_bf16_bits(z1);
      }
    }
  }
}

// Finish this warp's share of unit (kc, T): epilogue directly when the warp
// covered the whole tile, else publish the partial; the last contributor to
// the tile sums all partials in (k-chunk, warp) order and runs the epilogue.
template <int HD>
__device__ void gemv_finish(const Params& P, int layer, int st, const MatGeom& m, int kc, int T,
                            float acc0, float acc1, int64_t wg, int64_t W, const Misc& M) {
  const int lane = threadIdx.x & 31, t = lane & 3;
  const float sc = t < P.B ? M.escale[kc - M.kc_lo][t] : 0.f;
  const float v0 = acc0 * sc, v1 = acc1 * sc;
  const int64_t us = unit_start(m, kc, T), ue = us + chunk_groups(m, kc) - 1;
  const int64_t wf = owner_of(m.T, W, us), wl = owner_of(m.T, W, ue);
  if (m.Sk == 1 && wf == wl) {
    gemv_epilogue<HD>(P, layer, st, T, v0, v1, M);
    return;
  }
  const int64_t u = (int64_t)kc * m.NT + T;
  float2* part = reinterpret_cast<float2*>(P.gpart);
  part[(u * m.J + (wg - wf)) * 32 + lane] = make_float2(v0, v1);
  // contributors = warps with a non-empty range that own blocks of the tile
  // (with fewer blocks than warps, a warp owns at most one block)
  int ncontrib = 0;
  for (int k = 0; k < m.Sk; ++k) {
    const int64_t s0 = unit_start(m, k, T), e0 = s0 + chunk_groups(m, k) - 1;
    ncontrib += (int)(m.T >= W ? owner_of(m.T, W, e0) - owner_of(m.T, W, s0) + 1 : e0 - s0 + 1);
  }
  __syncwarp();
  uint32_t old = 0;
  if (lane == 0) {
    __threadfence();
    old = atomicAdd(P.cnt + T, 1u);
  }
  old = __shfl_sync(FULL, old, 0);
  if ((int)old != ncontrib - 1) return;
  __threadfence();
  float s0 = 0.f, s1 = 0.f;
  for (int k = 0; k < m.Sk; ++k) {
    const int64_t uk = (int64_t)k * m.NT + T;
    const int64_t a0 = unit_start(m, k, T), e0 = a0 + chunk_groups(m, k) - 1;
    const int64_t f0 = owner_of(m.T, W, a0), n0 = owner_of(m.T, W, e0) - f0 + 1;
    for (int64_t j = 0; j < n0; ++j) {
      if (range_lo(m.T, W, f0 + j) == range_lo(m.T, W, f0 + j + 1)) continue;  // empty range
      const float2 v = __ldcg(part + (uk * m.J + j) * 32 + lane);
      s0 += v.x;
      s1 += v.y;
    }
  }
  gemv_epilogue<HD>(P, layer, st, T, s0, s1, M);
  if (lane == 0) P.cnt[T] = 0;
}

// ------------------------------------------------------------------ GEMV stage
template <int HD, int WT>
__device__ bool stage_gemv(const Params& P, int layer, int st, Ring& R, Cursor& prod, int64_t wg,
                           int64_t W, uint8_t* smem, Misc& M, uint64_t policy) {
  const MatGeom& m = P.mg[stage_mat(st)];
  gemv_prologue<HD, WT>(P, layer, st, m, W, smem, M);
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int B = P.B, B2 = 2 * B;
  const int64_t lo = range_lo(m.T, W, wg), hi = range_lo(m.T, W, wg + 1);
  if (lo >= hi) return true;
  const uint32_t xf_base = smem_addr(smem + SM_SCR);
  const float* Sx = reinterpret_cast<const float*>(smem + SM_SCR + XF_BYTES);
  const int kc_lo = M.kc_lo;
  int kc, T, gi;
  block_coord(m, lo, kc, T, gi);
  int gk = chunk_groups(m, kc);
  float acc0 = 0.f, acc1 = 0.f;
  float cb[4] = {0.f, 0.f, 0.f, 0.f};  // bf16 path: fragment accumulators
  const int per = WT == DDL_W_INT4 ? BLKS_PER_SLOT : BF16_BLKS_PER_SLOT;
  for (int64_t b = lo; b < hi; b += per) {
    const int nb = (int)(hi - b < per ? hi - b : per);
    const uint32_t slot = R.slot(R.n_done);
    if (!mbar_wait_warp(R.bar(R.n_done), R.parity(R.n_done), P.ctrl + 1)) {
      M.abort = 1;
      return false;
    }
    for (int i = 0; i < nb; ++i) {
      const int kcl = kc - kc_lo;
      const uint32_t xfa = xf_base + (uint32_t)(((((kcl * GC + gi) * 4) * B2 + g) * 4 + t) * 8);
      if (WT == DDL_W_INT4) {
        const uint4 wv = lds128(slot + i * BLK_BYTES + lane * 16);
        const uint32_t sc = lds32(slot + BLKS_PER_SLOT * BLK_BYTES + i * SCL_BYTES + g * 4);
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w = ws[j], w8 = w >> 8;
          const uint32_t a0 = lop3_merge(w, 0x000F000Fu, 0x64086408u);
          const uint32_t a1 = lop3_merge(w, 0x00F000F0u, 0x64806480u);
          const uint32_t a2 = lop3_merge(w8, 0x000F000Fu, 0x64086408u);
          const uint32_t a3 = lop3_merge(w8, 0x00F000F0u, 0x64806480u);
          uint2 bf = make_uint2(0u, 0u);
          if (g < B2) bf = lds64(xfa + j * B2 * 32);
          mma_f16(c, a0, a1, a2, a3, bf.x, bf.y);
        }
        // rows g hold 1024 + (q+8), rows g+8 hold 1024 + 16 (q+8):
        // sum q x = v - 1032 Sx  and  (v - 1152 Sx) / 16
        const float sx = t < B ? Sx[(kcl * GC + gi) * MAX_B + t] : 0.f;
        acc0 = fmaf(bf16lo_f32(sc), (c[0] + c[1]) - 1032.f * sx, acc0);
        acc1 = fmaf(bf16hi_f32(sc) * 0.0625f, (c[2] + c[3]) - 1152.f * sx, acc1);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 av = lds128(slot + i * BF16_BLK_BYTES + j * 512 + lane * 16);
          uint2 bf = make_uint2(0u, 0u);
          if (g < B2) bf = lds64(xfa + j * B2 * 32);
          mma_bf16(cb, av.x, av.y, av.z, av.w, bf.x, bf.y);
        }
      }
      if (++gi == gk) {
        if (WT != DDL_W_INT4) {
          acc0 = cb[0] + cb[1];
          acc1 = cb[2] + cb[3];
          cb[0] = cb[1] = cb[2] = cb[3] = 0.f;
        }
        gemv_finish<HD>(P, layer, st, m, kc, T, acc0, acc1, wg, W, M);
        acc0 = acc1 = 0.f;
        gi = 0;
        if (++T == m.NT) {
          T = 0;
          ++kc;
          gk = kc < m.Sk ? chunk_groups(m, kc) : 0;
        }
      }
    }
    ring_advance<HD>(P, R, prod, wg, W, lane, policy);
  }
  if (gi != 0) {
    if (WT != DDL_W_INT4) {
      acc0 = cb[0] + cb[1];
      acc1 = cb[2] + cb[3];
    }
    gemv_finish<HD>(P, layer, st, m, kc, T, acc0, acc1, wg, W, M);
  }
  return true;
}

// ------------------------------------------------------------------ attention
// Merge n softmax states (m, l, o) into `out` (fp32 records of GH*(hd+2)).
template <int HD>
__device__ void merge_records(const float* const* recs, int n, float* out, int GH) {
  const int lane = threadIdx.x & 31;
  for (int h = lane; h < GH; h += 32) {
    float mx = -INFINITY;
    for (int k = 0; k < n; ++k) mx = fmaxf(mx, recs[k][GH * HD + h]);
    float l = 0.f;
    for (int k = 0; k < n; ++k) l += exp2f(recs[k][GH * HD + h] - mx) * recs[k][GH * HD + GH + h];
    out[GH * HD + h] = mx;
    out[GH * HD + GH + h] = l;
  }
  for (int e = lane; e < GH * HD; e += 32) {
    const int h = e / HD;
    float mx = -INFINITY;
    for (int k = 0; k < n; ++k) mx = fmaxf(mx, recs[k][GH * HD + h]);
    float o = 0.f;
    for (int k = 0; k < n; ++k) o += exp2f(recs[k][GH * HD + h] - mx) * recs[k][e];
    out[e] = o;
  }
}

template <int HD>
__device__ bool stage_att(const Params& P, int layer, Ring& R, Cursor& prod, int64_t wg, int64_t W,
                          uint8_t* smem, Misc& M, uint64_t policy) {
  constexpr int ROWB = HD * 2 + 16, KS = HD / 16, NB = HD / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int GH = P.GH, REC = GH * (HD + 2), nt = P.nt_att;
  const int64_t Ta = (int64_t)P.B * P.Hkv * nt, C = gridDim.x;
  const LayerDev& Ld = P.layers[layer];
  float* recs = reinterpret_cast<float*>(smem + SM_SCR);
  int64_t lo, hi;
  att_range(P, lo, hi);
  const float qscale = 1.4426950408889634f / sqrtf((float)HD);  // log2(e) / sqrt(hd)
  int nseg = 0;
  int64_t first_seq = -1, cur = -1;
  uint32_t qh[KS][2], ql[KS][2];
  float mrun = -INFINITY, lrun = 0.f;
  float o[NB][4];
  bool ok = true;

  auto flush = [&](bool at_end) {
    float ls = lrun + __shfl_xor_sync(FULL, lrun, 1);
    ls += __shfl_xor_sync(FULL, ls, 2);
    float* rec;
    if (nseg == 1) rec = recs + (warp * 2 + 0) * REC;
    else if (at_end) rec = recs + (warp * 2 + 1) * REC;
    else rec = P.apart + (cur * P.J_att + (blockIdx.x - owner_of(Ta, C, cur * nt))) * REC;
    if (g < GH) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        rec[g * HD + 8 * nb + 2 * t] = o[nb][0];
        rec[g * HD + 8 * nb + 2 * t + 1] = o[nb][1];
      }
      if (t == 0) {
        rec[GH * HD + g] = mrun;
        rec[GH * HD + GH + g] = ls;
      }
    }
  };

  for (int64_t it = lo; it < hi && ok; ++it) {
    const int64_t seq = it / nt;
    const int i = (int)(it % nt);
    if (seq != cur) {
      if (cur >= 0) flush(false);
      cur = seq;
      ++nseg;
      if (first_seq < 0) first_seq = seq;
      const int b = (int)(seq / P.Hkv), kvh = (int)(seq % P.Hkv);
      const float* qp = P.q + (int64_t)b * P.Hq * HD + (int64_t)(kvh * GH + g) * HD;
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (g < GH) {
          v[0] = __ldcg(qp + 16 * j + 2 * t) * qscale;
          v[1] = __ldcg(qp + 16 * j + 2 * t + 1) * qscale;
          v[2] = __ldcg(qp + 16 * j + 2 * t + 8) * qscale;
          v[3] = __ldcg(qp + 16 * j + 2 * t + 9) * qscale;
        }
        float h[4], l[4];
        for (int e = 0; e < 4; ++e) {
          h[e] = __bfloat162float(__float2bfloat16_rn(v[e]));
          l[e] = v[e] - h[e];
        }
        qh[j][0] = pack_bf16x2(h[0], h[1]);
        qh[j][1] = pack_bf16x2(h[2], h[3]);
        ql[j][0] = pack_bf16x2(l[0], l[1]);
        ql[j][1] = pack_bf16x2(l[2], l[3]);
      }
      mrun = -INFINITY;
      lrun = 0.f;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
    }
    const uint32_t ks = R.slot(R.n_done), vs = R.slot(R.n_done + 1);
    if (!mbar_wait_warp(R.bar(R.n_done), R.parity(R.n_done), P.ctrl + 1) ||
        !mbar_wait_warp(R.bar(R.n_done + 1), R.parity(R.n_done + 1), P.ctrl + 1)) {
      M.abort = 1;
      ok = false;
      break;
    }
    if (i == nt - 1) {  // the tile holding the new token: its row from the cache, zero rows after it
      const int rnew = (int)(P.pos - 16 * (int64_t)i);
      const int b = (int)(seq / P.Hkv), kvh = (int)(seq % P.Hkv);
      const int64_t ro = (((int64_t)b * P.Hkv + kvh) * P.s_max + P.pos) * HD;
      if (lane < HD / 8) sts128(ks + rnew * ROWB + lane * 16, ldcg_u128(Ld.kc + ro + lane * 8));
      else if (lane >= 16 && lane < 16 + HD / 8)
        sts128(vs + rnew * ROWB + (lane - 16) * 16, ldcg_u128(Ld.vc + ro + (lane - 16) * 8));
      const int nz = (15 - rnew) * (HD / 8);
      for (int z = lane; z < 2 * nz; z += 32) {
        const int zz = z % nz, row = rnew + 1 + zz / (HD / 8), col = zz % (HD / 8);
        sts128((z < nz ? ks : vs) + row * ROWB + col * 16, make_uint4(0u, 0u, 0u, 0u));
      }
      __syncwarp();
    }
    // scores S[head g][keys 8n + 2t, +1] = (q * log2e / sqrt(hd)) . K
    float s[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int jj = 0; jj < KS; jj += 2) {
        const int mat = lane >> 3, r = lane & 7;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ks + (8 * n + r) * ROWB + (16 * (jj + (mat >> 1)) + 8 * (mat & 1)) * 2, b0, b1, b2, b3);
        mma_bf16(s[n], qh[jj][0], 0u, qh[jj][1], 0u, b0, b1);
        mma_bf16(s[n], ql[jj][0], 0u, ql[jj][1], 0u, b0, b1);
        mma_bf16(s[n], qh[jj + 1][0], 0u, qh[jj + 1][1], 0u, b2, b3);
        mma_bf16(s[n], ql[jj + 1][0], 0u, ql[jj + 1][1], 0u, b2, b3);
      }
    }
    // online softmax over this tile
    float mt = -INFINITY;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int64_t key = 16 * (int64_t)i + 8 * n + 2 * t + e;
        if (key > P.pos) s[n][e] = -INFINITY;
        mt = fmaxf(mt, s[n][e]);
      }
    mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 2));
    const float mnew = fmaxf(mrun, mt);
    const float alpha = exp2f(mrun - mnew);
    float p[2][2];
    float psum = 0.f;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[n][e] = exp2f(s[n][e] - mnew);
        psum += p[n][e];
      }
    lrun = lrun * alpha + psum;
    mrun = mnew;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      o[nb][0] *= alpha;
      o[nb][1] *= alpha;
    }
    float ph[2][2], pl[2][2];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        ph[n][e] = __bfloat162float(__float2bfloat16_rn(p[n][e]));
        pl[n][e] = p[n][e] - ph[n][e];
      }
    const uint32_t pa0 = pack_bf16x2(ph[0][0], ph[0][1]), pa2 = pack_bf16x2(ph[1][0], ph[1][1]);
    const uint32_t pb0 = pack_bf16x2(pl[0][0], pl[0][1]), pb2 = pack_bf16x2(pl[1][0], pl[1][1]);
    // o[head g][d 8nb + 2t, +1] += P V
#pragma unroll
    for (int nb = 0; nb < NB; nb += 2) {
      const int mat = lane >> 3, r = lane & 7;
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vs + (8 * (mat & 1) + r) * ROWB + 8 * (nb + (mat >> 1)) * 2, b0, b1, b2, b3);
      mma_bf16(o[nb], pa0, 0u, pa2, 0u, b0, b1);
      mma_bf16(o[nb], pb0, 0u, pb2, 0u, b0, b1);
      mma_bf16(o[nb + 1], pa0, 0u, pa2, 0u, b2, b3);
      mma_bf16(o[nb + 1], pb0, 0u, pb2, 0u, b2, b3);
    }
    ring_advance<HD>(P, R, prod, wg, W, lane, policy);
    ring_advance<HD>(P, R, prod, wg, W, lane, policy);
  }
  if (ok && nseg > 0) flush(true);
  if (lane == 0) {
    M.seg_n[warp] = ok ? nseg : 0;
    M.seg_first[warp] = first_seq;
    M.seg_last[warp] = cur;
  }
  __syncthreads();
  if (M.abort) return false;
  // CTA merge: the warp where a sequence's run starts merges the run
  auto chain = [&](int64_t seq, int rec_idx, bool continues) {
    const float* list[NW + 1];
    int n = 0;
    list[n++] = recs + (warp * 2 + rec_idx) * REC;
    if (continues) {
      for (int v = warp + 1; v < NW; ++v) {
        if (M.seg_n[v] == 0) continue;
        if (M.seg_first[v] != seq) break;
        list[n++] = recs + (v * 2 + 0) * REC;
        if (M.seg_n[v] > 1) break;
      }
    }
    float* out = P.apart + (seq * P.J_att + (blockIdx.x - owner_of(Ta, C, seq * nt))) * REC;
    merge_records<HD>(list, n, out, GH);
  };
  const int ns = M.seg_n[warp];
  if (ns > 0) {
    bool owner = true;
    for (int v = warp - 1; v >= 0; --v) {
      if (M.seg_n[v] == 0) continue;
      owner = M.seg_last[v] != first_seq;
      break;
    }
    if (owner) chain(first_seq, 0, ns == 1);
    if (ns > 1) chain(cur, 1, true);
  }
  return true;
}

// Merge the CTA partials of each (sequence, head) into attn [B][Hq*hd].
template <int HD>
__device__ void stage_comb(const Params& P, int64_t wg, int64_t W) {
  const int lane = threadIdx.x & 31;
  const int GH = P.GH, REC = GH * (HD + 2), nt = P.nt_att;
  const int64_t Ta = (int64_t)P.B * P.Hkv * nt, C = gridDim.x;
  const int64_t items = (int64_t)P.B * P.Hq * (HD / 32);
  for (int64_t it = wg; it < items; it += W) {
    const int qd = (int)(it % (HD / 32));
    const int h = (int)((it / (HD / 32)) % P.Hq);
    const int b = (int)(it / (HD / 32) / P.Hq);
    const int64_t seq = (int64_t)b * P.Hkv + h / GH;
    const int hl = h % GH, d = qd * 32 + lane;
    const int64_t cf = owner_of(Ta, C, seq * nt), cl = owner_of(Ta, C, seq * nt + nt - 1);
    float mx = -INFINITY, l = 0.f, o = 0.f;
    for (int64_t jc = 0; jc <= cl - cf; ++jc) {
      if (range_lo(Ta, C, cf + jc) == range_lo(Ta, C, cf + jc + 1)) continue;  // CTA with no tiles
      const float* rec = P.apart + (seq * P.J_att + jc) * REC;
      const float m = __ldcg(rec + GH * HD + hl), lj = __ldcg(rec + GH * HD + GH + hl);
      const float oj = __ldcg(rec + hl * HD + d);
      const float mn = fmaxf(mx, m), a0 = exp2f(mx - mn), a1 = exp2f(m - mn);
      l = l * a0 + lj * a1;
      o = o * a0 + oj * a1;
      mx = mn;
    }
    P.attn[(int64_t)b * P.Hq * HD + (int64_t)h * HD + d] = o / l;
  }
}

// ------------------------------------------------------------------ grid barrier
__device__ bool grid_sync(const Params& P, uint32_t target, Misc& M) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(P.ctrl, 1u);
    const uint64_t t0 = globaltimer();
    while (ld_acquire_gpu(P.ctrl) < target) {
      __nanosleep(64);
      if (globaltimer() - t0 > WAIT_LIMIT_NS) {
        atomicExch(P.ctrl + 1, STATUS_TIMEOUT);
        M.abort = 1;
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();
  return !M.abort;
}

// ------------------------------------------------------------------ the kernel
template <int HD, int WT>
__global__ void __launch_bounds__(NTHREADS, 1) decode_kernel(const __grid_constant__ Params P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t W = (int64_t)gridDim.x * NW, wg = (int64_t)blockIdx.x * NW + warp;
  Misc& M = *reinterpret_cast<Misc*>(smem + SM_MISC);
  Ring R;
  R.slot0 = smem_addr(smem + SM_RING + warp * DEPTH * SLOT_BYTES);
  R.bar0 = smem_addr(smem + SM_BARS + warp * DEPTH * 8);
  R.n_issued = R.n_done = 0;
  if (lane < DEPTH) mbar_init(R.bar0 + lane * 8, 1);
  if (threadIdx.x == 0) M.abort = 0;
  mbar_init_fence();
  __syncthreads();
  const uint64_t policy = policy_evict_first();
  Cursor prod;
  prod.s = P.stage_begin;
  cursor_range(P, prod.s, wg, W, prod.pos, prod.end);
  for (int k = 0; k < DEPTH; ++k) {
    SlotDesc d;
    if (!cursor_next(P, prod, wg, W, d)) break;
    issue_slot<HD>(P, d, R.slot(R.n_issued), R.bar(R.n_issued), lane, policy);
    R.n_issued++;
  }
  bool ok = true;
  for (int s = P.stage_begin; s < P.stage_end && ok; ++s) {
    if (s != P.stage_begin && P.cooperative) {
      if (!grid_sync(P, (uint32_t)(s - P.stage_begin) * gridDim.x, M)) {
        ok = false;
        break;
      }
    }
    const int layer = s / NSTAGE, st = s % NSTAGE;
    if (st == ST_ATT) {
      ok = stage_att<HD>(P, layer, R, prod, wg, W, smem, M, policy);
    } else if (st == ST_COMB) {
      stage_comb<HD>(P, wg, W);
    } else {
      stage_gemv<HD, WT>(P, layer, st, R, prod, wg, W, smem, M, policy);
    }
    __syncthreads();
    if (M.abort) ok = false;
  }
  if (!ok) {  // let this warp's copies in flight land before the CTA exits (bounded)
    for (uint32_t n = R.n_done; n < R.n_issued; ++n)
      if (!mbar_wait_warp(R.bar(n), R.parity(n), P.ctrl + 1)) break;
  }
}

// ------------------------------------------------------------------ host runtime
static char g_cuda_err[256] = "";
void set_cuda_error(cudaError_t e) {
  snprintf(g_cuda_err, sizeof g_cuda_err, "%s", cudaGetErrorString(e));
}

struct DevInfo {
  int sms = 0, coop = 0, ok = 0;
};
static std::mutex g_mu;
static DevInfo g_dev[64];
static int g_launch_mode = 0;  // 0 automatic, 1 one launch per stage

template <int HD, int WT>
static int prepare_kernel() {
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (done[dev]) return DDL_OK;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<HD, WT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SM_TOTAL);
  if (e != cudaSuccess) return cuda_status(e);
  done[dev] = true;
  return DDL_OK;
}

static int device_info(DevInfo& out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  std::lock_guard<std::mutex> lk(g_mu);
  if (dev < 0 || dev >= 64) return DDL_ERR_UNSUPPORTED;
  if (!g_dev[dev].ok) {
    int sms = 0, coop = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_status(e);
    if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess)
      return cuda_status(e);
    g_dev[dev].sms = sms;
    g_dev[dev].coop = coop;
    g_dev[dev].ok = 1;
  }
  out = g_dev[dev];
  return DDL_OK;
}

struct WsLayout {
  int64_t ctrl, cnt, gpart, apart, Z, q, attn, y, a, total;
};

static int64_t att_J(int64_t seqs, int64_t nt, int64_t C) {
  const int64_t Ta = seqs * nt;
  int64_t J = 1;
  for (int64_t s = 0; s < seqs; ++s) {
    const int64_t n = owner_of(Ta, C, s * nt + nt - 1) - owner_of(Ta, C, s * nt) + 1;
    if (n > J) J = n;
  }
  return J;
}

static void ws_layout(const ddl_shape& s, int B, int64_t s_max, int C, const MatGeom mg[4],
                      WsLayout& w) {
  const int64_t Nq = (int64_t)s.H_q * s.head_dim, GH = s.H_q / s.H_kv;
  // attention partial slot of a sequence = CTA index - the sequence's first CTA;
  // with fewer tiles than CTAs that span includes CTAs without tiles, so it is
  // bounded by the grid, not by the tile count
  const int64_t Jatt = C;
  int64_t gpart = 0, ntmax = 0;
  for (int k = 0; k < 4; ++k) {
    const int64_t u = (int64_t)mg[k].Sk * mg[k].NT * mg[k].J * 32 * 2 * 4;
    if (u > gpart) gpart = u;
    if (mg[k].NT > ntmax) ntmax = mg[k].NT;
  }
  int64_t off = 0;
  w.ctrl = off;  off = align256(off + 256);
  w.cnt = off;   off = align256(off + ntmax * 4);
  w.gpart = off; off = align256(off + gpart);
  w.apart = off; off = align256(off + (int64_t)B * s.H_kv * (Jatt + 1) * GH * (s.head_dim + 2) * 4);
  w.Z = off;     off = align256(off + 2 * (int64_t)B * s.D * 4);
  w.q = off;     off = align256(off + (int64_t)B * Nq * 4);
  w.attn = off;  off = align256(off + (int64_t)B * Nq * 4);
  w.y = off;     off = align256(off + (int64_t)B * s.D * 4);
  w.a = off;     off = align256(off + (int64_t)B * s.d_ff * 4);
  w.total = off;
}

static int plan(const ddl_shape* s, int wtype, int B, int64_t s_max, int C, MatGeom mg[4],
                WsLayout& w) {
  make_geoms(*s, wtype, mg);
  for (int k = 0; k < 4; ++k) mg[k].J = max_warps_per_unit(mg[k], (int64_t)C * NW);
  ws_layout(*s, B, s_max, C, mg, w);
  return DDL_OK;
}

static int decode(const ddl_shape* s, ddl_wtype wtype, const ddl_layer_w* layers, const ddl_kv* kv,
                  int32_t L, int32_t B, int64_t pos, const float* resid_in, const uint16_t* x_bf16,
                  float* resid_out, uint16_t* out_bf16, void* workspace, size_t ws_bytes,
                  void* stream) {
  int st = check_shape(s);
  if (st) return st;
  if (!layers || !kv || L <= 0 || !workspace) return !workspace ? DDL_ERR_WORKSPACE : DDL_ERR_ARG;
  if (B < 1 || B > MAX_B) return DDL_ERR_UNSUPPORTED;
  if (wtype != DDL_W_INT4 && wtype != DDL_W_BF16) return DDL_ERR_UNSUPPORTED;
  if (!resid_in && !x_bf16) return DDL_ERR_ARG;
  const int64_t s_max = kv[0].s_max;
  if (pos < 0 || pos >= s_max) return DDL_ERR_POS;
  for (int l = 0; l < L; ++l) {
    if (!layers[l].packed || !layers[l].norm1 || !layers[l].norm2 || !kv[l].k || !kv[l].v)
      return DDL_ERR_ARG;
    if (kv[l].s_max != s_max) return DDL_ERR_ARG;
    if (!aligned16(layers[l].packed) || !aligned16(layers[l].norm1) || !aligned16(layers[l].norm2) ||
        !aligned16(kv[l].k) || !aligned16(kv[l].v))
      return DDL_ERR_ALIGN;
  }
  if (!aligned16(workspace) || (resid_in && !aligned16(resid_in)) || (x_bf16 && !aligned16(x_bf16)) ||
      (resid_out && !aligned16(resid_out)) || (out_bf16 && !aligned16(out_bf16)))
    return DDL_ERR_ALIGN;
  DevInfo di;
  if ((st = device_info(di))) return st;
  const int C = di.sms;
  Params P;
  memset(&P, 0, sizeof P);
  WsLayout w;
  plan(s, wtype, B, s_max, C, P.mg, w);
  for (int k = 0; k < 4; ++k)  // a CTA's share of a stream must touch at most two k-chunks
    if ((P.mg[k].T + C - 1) / C > (int64_t)P.mg[k].NT * P.mg[k].Gc) return DDL_ERR_UNSUPPORTED;
  if ((int64_t)ws_bytes < w.total) return DDL_ERR_WORKSPACE;
  const int HD = s->head_dim;
  st = HD == 128 ? (wtype == DDL_W_INT4 ? prepare_kernel<128, DDL_W_INT4>() : prepare_kernel<128, DDL_W_BF16>())
                 : (wtype == DDL_W_INT4 ? prepare_kernel<64, DDL_W_INT4>() : prepare_kernel<64, DDL_W_BF16>());
  if (st) return st;
  uint8_t* ws = (uint8_t*)workspace;
  P.D = s->D; P.Hq = s->H_q; P.Hkv = s->H_kv; P.hd = HD; P.dff = s->d_ff; P.B = B;
  P.GH = s->H_q / s->H_kv; P.eps = s->eps; P.wtype = wtype; P.rope_base = s->rope_base;
  P.pos = pos; P.s_max = s_max;
  P.nt_att = (int32_t)((pos + 1 + 15) / 16);
  P.J_att = (int32_t)att_J((int64_t)B * s->H_kv, P.nt_att, C);
  P.resid_in = resid_in; P.x_bf16 = x_bf16; P.resid_out = resid_out; P.out_bf16 = out_bf16;
  P.ctrl = (uint32_t*)(ws + w.ctrl); P.cnt = (uint32_t*)(ws + w.cnt);
  P.gpart = (float*)(ws + w.gpart); P.apart = (float*)(ws + w.apart); P.Z = (float*)(ws + w.Z);
  P.q = (float*)(ws + w.q); P.attn = (float*)(ws + w.attn); P.y = (float*)(ws + w.y);
  P.a = (float*)(ws + w.a);
  cudaStream_t cs = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(ws, 0, (size_t)w.gpart, cs);  // barrier, status, tile counters
  if (e != cudaSuccess) return cuda_status(e);
  const bool coop = di.coop && g_launch_mode == 0;
  void* fn = HD == 128 ? (wtype == DDL_W_INT4 ? (void*)decode_kernel<128, DDL_W_INT4> : (void*)decode_kernel<128, DDL_W_BF16>)
                       : (wtype == DDL_W_INT4 ? (void*)decode_kernel<64, DDL_W_INT4> : (void*)decode_kernel<64, DDL_W_BF16>);
  for (int l0 = 0; l0 < L; l0 += MAX_LAYERS) {
    const int nL = L - l0 < MAX_LAYERS ? L - l0 : MAX_LAYERS;
    P.L = nL;
    P.l0 = l0;
    P.final_last = (l0 + nL == L);
    for (int l = 0; l < nL; ++l) {
      P.layers[l].packed = (const uint8_t*)layers[l0 + l].packed;
      P.layers[l].norm1 = layers[l0 + l].norm1;
      P.layers[l].norm2 = layers[l0 + l].norm2;
      P.layers[l].kc = kv[l0 + l].k;
      P.layers[l].vc = kv[l0 + l].v;
    }
    if (coop) {
      if (l0 > 0 && (e = cudaMemsetAsync(ws + w.ctrl, 0, 4, cs)) != cudaSuccess) return cuda_status(e);
      P.stage_begin = 0;
      P.stage_end = nL * NSTAGE;
      P.cooperative = 1;
      void* args[] = {&P};
      e = cudaLaunchCooperativeKernel(fn, dim3(C), dim3(NTHREADS), args, SM_TOTAL, cs);
      if (e != cudaSuccess) return cuda_status(e);
    } else {
      P.cooperative = 0;
      for (int sidx = 0; sidx < nL * NSTAGE; ++sidx) {
        P.stage_begin = sidx;
        P.stage_end = sidx + 1;
        void* args[] = {&P};
        e = cudaLaunchKernel(fn, dim3(C), dim3(NTHREADS), args, SM_TOTAL, cs);
        if (e != cudaSuccess) return cuda_status(e);
      }
    }
  }
  return DDL_OK;
}

}  // namespace ddl

using namespace ddl;

extern "C" size_t ddl_workspace_bytes(const ddl_shape* shape, int32_t B, int64_t s_max) {
  if (check_shape(shape) || B < 1 || B > MAX_B || s_max < 1) return 0;
  DevInfo di;
  if (device_info(di)) return 0;
  MatGeom mg[4];
  WsLayout w;
  plan(shape, DDL_W_INT4, B, s_max, di.sms, mg, w);
  WsLayout w2;
  MatGeom mg2[4];
  plan(shape, DDL_W_BF16, B, s_max, di.sms, mg2, w2);
  return (size_t)(w.total > w2.total ? w.total : w2.total);
}

extern "C" int ddl_workspace_view(const ddl_shape* shape, int32_t B, int64_t s_max,
                                  ddl_ws_view* out) {
  int st = check_shape(shape);
  if (st) return st;
  if (!out || B < 1 || B > MAX_B || s_max < 1) return DDL_ERR_ARG;
  DevInfo di;
  if ((st = device_info(di))) return st;
  MatGeom mg[4];
  WsLayout w;
  plan(shape, DDL_W_INT4, B, s_max, di.sms, mg, w);
  out->q = (size_t)w.q;
  out->attn = (size_t)w.attn;
  out->y = (size_t)w.y;
  out->a = (size_t)w.a;
  out->status = (size_t)w.ctrl + 4;
  return DDL_OK;
}

extern "C" int ddl_layer_decode(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layer,
                                const ddl_kv* kv, int32_t B, int64_t pos, const float* resid_in,
                                const uint16_t* x_bf16, float* resid_out, uint16_t* out_bf16,
                                void* workspace, size_t ws_bytes, void* stream) {
  return decode(shape, wtype, layer, kv, 1, B, pos, resid_in, x_bf16, resid_out, out_bf16,
                workspace, ws_bytes, stream);
}

extern "C" int ddl_stack_decode(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layers,
                                const ddl_kv* kv, int32_t L, int32_t B, int64_t pos,
                                const float* resid_in, const uint16_t* x_bf16, float* resid_out,
                                uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream) {
  return decode(shape, wtype, layers, kv, L, B, pos, resid_in, x_bf16, resid_out, out_bf16,
                workspace, ws_bytes, stream);
}

extern "C" int ddl_set_launch_mode(int32_t mode) {
  if (mode != 0 && mode != 1) return DDL_ERR_ARG;
  g_launch_mode = mode;
  return DDL_OK;
}

extern "C" int ddl_read_device_status(const void* workspace, const ddl_shape* shape, int32_t B,
                                      int64_t s_max, int32_t* status_out, void* stream) {
  if (!workspace || !status_out) return DDL_ERR_ARG;
  ddl_ws_view v;
  int st = ddl_workspace_view(shape, B, s_max, &v);
  if (st) return st;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e);
  uint32_t word = 0;
  e = cudaMemcpy(&word, (const uint8_t*)workspace + v.status, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  *status_out = (int32_t)word;
  return DDL_OK;
}

extern "C" const char* ddl_status_string(int status) {
  switch (status) {
    case DDL_OK: return "ok";
    case DDL_ERR_SHAPE: return "unsupported shape";
    case DDL_ERR_POS: return "position outside the KV cache";
    case DDL_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case DDL_ERR_WORKSPACE: return "workspace missing or too small";
    case DDL_ERR_UNSUPPORTED: return "unsupported weight type, batch or device";
    case DDL_ERR_CUDA: return "CUDA runtime error";
    case DDL_ERR_TIMEOUT: return "a bounded device wait gave up";
    case DDL_ERR_ARG: return "invalid argument";
    default: return "unknown status";
  }
}

extern "C" const char* ddl_last_cuda_error(void) { return g_cuda_err; }
