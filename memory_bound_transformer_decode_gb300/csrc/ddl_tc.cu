// ddl_tc.cu -- the batched decode step's weight stages on the tcgen05 tensor
// cores (batches of 16-64 sequences with INT4 weights, 5-64 with bf16), where
// the step's matrix products are real dense contractions ("把基础打牢"
// primer §1.3: batching raises the intensity; roofline reply §七).
//
// GEMM kernel (one launch per weight stage): a CTA takes units of 128 weight
// rows (eight of the packed stream's 16-row tiles) by a range of 64-wide
// groups of the input dimension.  Warp 0 copies each group's eight packed
// blocks and the group's B-operand image (the activations as two fp16 limbs, laid
// out as the tensor core reads them) into a ring of shared-memory stages with
// TMA bulk copies; three warpgroups take the groups in turn, expand the 4-bit
// codes (or bf16 weights) in registers to fp16 and store them into tensor
// memory as the A operand (one 32-lane quarter per warp; the tcgen05.st
// 16x256b shape takes the tensor-core fragment registers as they are); one
// thread of warp 1 issues the tcgen05.mma of the group's four 16-wide slices
// into an fp32 accumulator in tensor memory and commits them to mbarriers
// that hand the A buffer back.  A stage goes back to the copy warp once its
// MMAs have completed and every expansion warp has released it: each of them
// waits for every stage in turn, also those without a group of its own, so
// that no stage's barrier runs a phase ahead of a reader (a parity wait on a
// barrier two phases behind would return at once).  At a unit's end the last
// warpgroup reads the accumulator (tcgen05.ld), combines the two limb columns
// of each sequence and stores the unit's partial sums.
//
// Epilogue kernel (one launch per stage): sums a stage's split-K partials in a
// fixed order and applies what the layer does to that stage's output (RMSNorm
// factor, RoPE, the K/V append, the residual adds, SwiGLU), and writes the
// B-operand image of the next GEMM's input (the activations times the next
// RMSNorm weight, as two fp16 limbs) with per-CTA sums of squares.
#include <math.h>

#include <cuda_fp16.h>

#include "ddl_device.cuh"
#include "ddl_internal.h"
#include "ddl_tc.h"

namespace ddl {

namespace {

// GEMM CTA: warp 0 copies, warp 1 issues the MMAs, NDW warpgroups from warp
// 4 on expand A, the last warpgroup reads the accumulators out.
constexpr int NDW = 3;
constexpr int GT = 32 * (4 + 4 * NDW + 4);
constexpr int MAX_STAGES = 8;
constexpr int MAX_NA = 12;       // A buffers in tensor memory (barrier slots)
constexpr int TMEM_COLS = 512;
constexpr int A_COLS = 32;       // one group of A: four 16-wide slices of 8 columns
constexpr int LBO = 128, SBO = 1024;  // B-operand image: k-cores of 8 x 16 B, 8 k-cores per column group of 8

struct TcGemm {
  int32_t N, NT, G, Sk, Gc, glast, NR, NP, B;
  uint32_t W, parts;             // (128-row tile, group) items NR * G, CTAs sharing them (the grid)
  uint32_t wbytes, stage_bytes;  // bytes of a stage's weights area (aligned), of a whole stage
  int32_t stages;                // shared-memory ring depth
  int32_t gs;                    // groups per ring stage (at most)
  int32_t na, nd;                // A buffers (32 columns each, from column 0), accumulators (after them)
  int32_t dstride;               // columns of an accumulator: NP + 16 (the read-out takes 16 at a time)
  const uint8_t* w;              // the matrix's block stream
  const uint8_t* xl;             // B-operand images, NP * 128 bytes per group
  float* part;                   // [S][B][N] partial sums, rows in the packed (tile) order
  const float* ss_in;            // QKV, gate/up: the epilogue CTAs' sums of squares of the stage input ...
  float* rfac;                   // ... reduced here to the RMSNorm factor per sequence (else NULL)
  int32_t ss_K;                  // the input's length
  float eps;
  uint32_t* status;
  uint64_t wait_ns;
};

__device__ __forceinline__ int64_t block_index(const TcGemm& P, int T, int g) {
  const int kc = g / P.Gc, gi = g - kc * P.Gc, gk = kc == P.Sk - 1 ? P.glast : P.Gc;
  return (int64_t)kc * P.NT * P.Gc + (int64_t)T * gk + gi;
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// fp16 code * scale of one 32-bit word of packed nibbles (the eight codes of
// rows g, g+8 at k 2t, 2t+1, 2t+8, 2t+9 of a 16-wide slice): r0 = row g,
// k (2t, 2t+1); r1 = row g, k (2t+8, 2t+9); r2, r3 the same for row g+8.
// (1032 + code) comes out exact from the fp16 pattern 0x6408 | (code ^ 8);
// minus 1032 gives the code, times the fp16 scale the exact product.
__device__ __forceinline__ void expand_int4(uint32_t w, __half2 s0, __half2 s1, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  const __half2 off = u2h(0x64086408u);
  const __half2 c0 = __hsub2(u2h(lop3_merge(w, 0x000F000Fu, 0x64086408u)), off);
  const __half2 c1 = __hsub2(u2h(lop3_merge(w >> 4, 0x000F000Fu, 0x64086408u)), off);
  const __half2 c2 = __hsub2(u2h(lop3_merge(w >> 8, 0x000F000Fu, 0x64086408u)), off);
  const __half2 c3 = __hsub2(u2h(lop3_merge(w >> 12, 0x000F000Fu, 0x64086408u)), off);
  r0 = h2u(__hmul2(c0, s0));
  r1 = h2u(__hmul2(c2, s0));
  r2 = h2u(__hmul2(c1, s1));
  r3 = h2u(__hmul2(c3, s1));
}
__device__ __forceinline__ uint32_t bf16pair_to_f16pair(uint32_t v) {
  return h2u(__floats2half2_rn(bf16lo_f32(v), bf16hi_f32(v)));
}

// A unit's k-range [g0, g1) is cut into ring stages of up to P.gs groups that
// stay inside one k-chunk, so that each tile's blocks of a stage are one
// contiguous run of the stream (one bulk copy per tile and stage).
__device__ __forceinline__ int stage_groups(const TcGemm& P, int g, int g1) {
  const int cend = (g / P.Gc + 1) * P.Gc;
  int e = g + P.gs;
  if (e > cend) e = cend;
  if (e > g1) e = g1;
  return e - g;
}

// A CTA's work: items [w, w1) of the (128-row tile, 64-wide group) order,
// tile-major, an equal share of all items; cut at tile edges into segments,
// each one accumulator's run and one split-K partial of its tile (slot: the
// CTA's index minus that of the first CTA holding part of the tile).
struct Seg {
  uint32_t w, w1;
  int r, g0, g1;
  __device__ __forceinline__ bool next(uint32_t G) {
    if (w >= w1) return false;
    r = (int)(w / G);
    g0 = (int)(w - (uint32_t)r * G);
    const uint32_t e = w1 < (uint32_t)(r + 1) * G ? w1 : (uint32_t)(r + 1) * G;
    g1 = g0 + (int)(e - w);
    w = e;
    return true;
  }
};
__device__ __forceinline__ Seg cta_work(const TcGemm& P) {
  Seg s;
  s.w = (uint32_t)range_lo(P.W, P.parts, blockIdx.x);
  s.w1 = (uint32_t)range_lo(P.W, P.parts, blockIdx.x + 1);
  return s;
}

template <int WT>
__global__ void __launch_bounds__(GT, 1) tc_gemm_kernel(const __grid_constant__ TcGemm P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr uint32_t BB = WT == DDL_W_INT4 ? QBLK_BYTES : BF16_BLK_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = P.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * P.stage_bytes);
  const uint32_t full0 = smem_addr(bars), empty0 = full0 + MAX_STAGES * 8;
  const int NA = P.na, ND = P.nd;
  const uint32_t D_COL0 = (uint32_t)NA * A_COLS;
  const uint32_t aready0 = empty0 + MAX_STAGES * 8, afree0 = aready0 + MAX_NA * 8;
  const uint32_t dready0 = afree0 + MAX_NA * 8, dfree0 = dready0 + 16, fin = dfree0 + 16;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * MAX_STAGES + 2 * MAX_NA + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + i * 8, 1);
      mbar_init(empty0 + i * 8, 1 + 4 * NDW);  // the MMA commit and each expansion warp
    }
    for (int i = 0; i < NA; ++i) {
      mbar_init(aready0 + i * 8, 4);
      mbar_init(afree0 + i * 8, 1);
    }
    for (int i = 0; i < ND; ++i) {
      mbar_init(dready0 + i * 8, 1);
      mbar_init(dfree0 + i * 8, 4);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
  }
  mbar_init_fence();
  __syncthreads();
  if (warp == 1) tmem_alloc(smem_addr(tslot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tslot;
  const uint32_t sbase = smem_addr(smem);
  pdl_wait();  // the previous kernel's operand images, and its reads of the partials this kernel writes
  auto fail = [&]() {
    if ((threadIdx.x & 31) == 0) atomicExch(P.status, STATUS_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {  // ------------------------------------------------ copies
    const uint64_t policy = policy_evict_first();
    uint32_t sc = 0;  // stages issued
    bool ok = true;
    for (Seg sg = cta_work(P); ok && sg.next((uint32_t)P.G);) {
      const int T0 = sg.r * 8, nt = P.NT - T0 < 8 ? P.NT - T0 : 8;
      const int g0 = sg.g0, g1 = sg.g1;
      for (int g = g0; g < g1; ++sc) {
        const int ng = stage_groups(P, g, g1);
        const uint32_t st = sc % NS, k = sc / NS;
        if (k > 0 && !mbar_wait_warp(empty0 + st * 8, (k - 1) & 1, P.status, P.wait_ns)) {
          fail();
          ok = false;
          break;
        }
        const uint32_t slot = sbase + st * P.stage_bytes;
        if (lane == 0) mbar_arrive_expect_tx(full0 + st * 8, (uint32_t)(nt * ng) * BB + (uint32_t)ng * P.NP * 128u);
        __syncwarp();
        if (lane < nt)  // tile T0 + lane, groups g .. g + ng - 1: one run of the stream
          bulk_g2s_evict_first(slot + lane * (P.gs * BB), P.w + block_index(P, T0 + lane, g) * BB, ng * BB,
                               full0 + st * 8, policy);
        if (lane == 8)
          bulk_g2s(slot + P.wbytes, P.xl + (int64_t)g * P.NP * 128, (uint32_t)ng * P.NP * 128u, full0 + st * 8);
        g += ng;
      }
      if (*abort_flag) ok = false;
    }
    // copies in flight land before the CTA leaves (bounded)
    if (lane == 0)
      for (uint32_t j = sc > (uint32_t)NS ? sc - NS : 0; j < sc; ++j)
        if (!mbar_wait_thread(full0 + (j % NS) * 8, (j / NS) & 1, P.wait_ns)) break;
  } else if (warp == 1) {  // ------------------------------------ MMA issue
    // the whole warp runs the loop (warp-uniform operands); one lane issues
    const uint32_t idesc = umma_idesc_f16(128, P.NP);
    const uint64_t xdesc0 = umma_sdesc(sbase + P.wbytes, LBO, SBO);  // stage 0's first group, slice 0
    const uint32_t gstep = (uint32_t)P.NP * 128u >> 4, sstep = P.stage_bytes >> 4;  // descriptor address units
    uint32_t sc = 0, it = 0, ui = 0;
    bool ok = true;
    for (Seg sg = cta_work(P); ok && sg.next((uint32_t)P.G); ++ui) {
      const int g0 = sg.g0, g1 = sg.g1;
      const uint32_t db = ui % ND, dk = ui / ND, dcol = tm + D_COL0 + db * P.dstride;
      if (dk > 0 && !mbar_wait_warp(dfree0 + db * 8, (dk - 1) & 1, P.status, P.wait_ns)) {
        fail();
        break;
      }
      tc_fence_after();
      bool first = true;
      for (int g = g0; g < g1 && ok; ++sc) {
        const int ng = stage_groups(P, g, g1);
        const uint32_t st = sc % NS, k = sc / NS;
        if (!mbar_wait_warp(full0 + st * 8, k & 1, P.status, P.wait_ns)) {
          fail();
          ok = false;
          break;
        }
        uint64_t xd = xdesc0 + (uint64_t)(st * sstep);
        for (int gi = 0; gi < ng; ++gi, ++it, xd += gstep) {
          const uint32_t ab = it % NA, ka = it / NA;
          if (!mbar_wait_warp(aready0 + ab * 8, ka & 1, P.status, P.wait_ns)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint32_t aa = tm + ab * A_COLS;
            umma_f16_ts(dcol, aa, xd, idesc, first ? 0u : 1u);
            umma_f16_ts(dcol, aa + 8, xd + (2 * LBO >> 4), idesc, 1u);
            umma_f16_ts(dcol, aa + 16, xd + (4 * LBO >> 4), idesc, 1u);
            umma_f16_ts(dcol, aa + 24, xd + (6 * LBO >> 4), idesc, 1u);
            umma_commit(afree0 + ab * 8);
          }
          __syncwarp();
          first = false;
        }
        if (!ok) break;
        if (elect_one()) umma_commit(empty0 + st * 8);
        __syncwarp();
        g += ng;
      }
      if (ok && elect_one()) umma_commit(dready0 + db * 8);
      __syncwarp();
    }
    // every MMA issued has completed before tensor memory is released
    if (elect_one()) umma_commit(fin);
    __syncwarp();
    mbar_wait_warp(fin, 0, P.status, P.wait_ns);
  } else if (warp == 3) {  // ----------------------------- RMSNorm factors
    // for the stage's epilogue, once per sequence instead of in each of its
    // CTAs: lane l sums CTAs l, l + 32, ... in that order, then a fixed tree
    if (P.rfac)
      for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
        float ss = 0.f;
#pragma unroll
        for (int c = lane; c < TC_EPI_CTAS; c += 32) ss += __ldcg(P.ss_in + c * P.B + b);
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) P.rfac[b] = 1.0f / sqrtf(ss / (float)P.ss_K + P.eps);
      }
  } else if (warp >= 4 && warp < 4 + 4 * NDW) {  // ------------------ A operand
    // expansion warpgroup d takes the CTA's groups it, it + NDW, ...; warp q
    // of it writes tensor-memory lanes 32 q .. 32 q + 31 (tiles 2q, 2q+1)
    const int d = (warp - 4) >> 2, q = warp & 3, g = lane >> 2;
    uint32_t sc = 0, it = 0;
    bool ok = true;
    for (Seg sg = cta_work(P); ok && sg.next((uint32_t)P.G);) {
      const int T0 = sg.r * 8, nt = P.NT - T0 < 8 ? P.NT - T0 : 8;
      const int g0 = sg.g0, g1 = sg.g1;
      for (int gs = g0; gs < g1 && ok; ++sc) {
        const int ng = stage_groups(P, gs, g1);
        const uint32_t st = sc % NS, k = sc / NS;
        const uint32_t slot = sbase + st * P.stage_bytes;
        // every stage, in order: the stage cannot be refilled before this
        // warp has released it, so this phase is the barrier's next one
        if (!mbar_wait_warp(full0 + st * 8, k & 1, P.status, P.wait_ns)) {
          fail();
          ok = false;
          break;
        }
        for (int gi = 0; gi < ng; ++gi, ++it) {
          if ((int)(it % NDW) != d) continue;
          const uint32_t ab = it % NA, ka = it / NA;
          if (ka > 0 && !mbar_wait_warp(afree0 + ab * 8, (ka - 1) & 1, P.status, P.wait_ns)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int tile = 2 * q + h;
            const uint32_t ta = tm + ((uint32_t)(32 * q + 16 * h) << 16) + ab * A_COLS;
            if (tile < nt) {
              const uint32_t blk = slot + tile * (P.gs * BB) + gi * BB;
              if (WT == DDL_W_INT4) {
                const uint4 wv = lds128(blk + lane * 16);
                const uint32_t sw = lds32(blk + BLK_BYTES + g * 4);
                const __half2 s0 = __float2half2_rn(bf16lo_f32(sw)), s1 = __float2half2_rn(bf16hi_f32(sw));
                uint32_t r[4][4];
                expand_int4(wv.x, s0, s1, r[0][0], r[0][1], r[0][2], r[0][3]);
                expand_int4(wv.y, s0, s1, r[1][0], r[1][1], r[1][2], r[1][3]);
                expand_int4(wv.z, s0, s1, r[2][0], r[2][1], r[2][2], r[2][3]);
                expand_int4(wv.w, s0, s1, r[3][0], r[3][1], r[3][2], r[3][3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) tmem_st_16x256b(ta + 8 * j, r[j][0], r[j][1], r[j][2], r[j][3]);
              } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {  // a0..a3 of the fragment: (g, lo k), (g+8, lo k), (g, hi k), (g+8, hi k)
                  const uint4 av = lds128(blk + j * 512 + lane * 16);
                  tmem_st_16x256b(ta + 8 * j, bf16pair_to_f16pair(av.x), bf16pair_to_f16pair(av.z),
                                  bf16pair_to_f16pair(av.y), bf16pair_to_f16pair(av.w));
                }
              }
            } else {  // rows past the matrix's end: zero
#pragma unroll
              for (int j = 0; j < 4; ++j) tmem_st_16x256b(ta + 8 * j, 0u, 0u, 0u, 0u);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_local(aready0 + ab * 8);
        }
        if (!ok) break;
        // this warp's reads of the stage's weights are done (their values
        // went into tensor memory above): the stage may be refilled
        __syncwarp();
        if (lane == 0) mbar_arrive_local(empty0 + st * 8);
        gs += ng;
      }
      if (*abort_flag) ok = false;
    }
  } else if (warp >= 4 + 4 * NDW) {  // --------------------------- read-out
    // the accumulator of each unit: row 32 q + lane, limb columns l * B + b (l = 0, 1)
    const int q = warp & 3;
    uint32_t ui = 0;
    for (Seg sg = cta_work(P); sg.next((uint32_t)P.G); ++ui) {
      const int rt = sg.r;
      const int s = (int)blockIdx.x - (int)owner32(P.W, P.parts, (uint32_t)rt * (uint32_t)P.G);
      const uint32_t db = ui % ND, dk = ui / ND;
      if (!mbar_wait_warp_nap(dready0 + db * 8, dk & 1, P.status, P.wait_ns, 500)) {  // a unit takes many us
        fail();
        break;
      }
      tc_fence_after();
      const int n = rt * 128 + 32 * q + lane;
      const uint32_t tr = tm + ((uint32_t)(32 * q) << 16) + D_COL0 + db * P.dstride;
      for (int b0 = 0; b0 < P.B; b0 += 16) {
        uint32_t v0[16], v1[16];
        tmem_ld_32x32b_x16(tr + b0, v0);
        tmem_ld_32x32b_x16(tr + P.B + b0, v1);
        tmem_ld_wait();
        if (n < P.N) {
          float* dst = P.part + (int64_t)s * P.B * P.N + n;  // [S][B][N]: the lanes' rows are consecutive
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (b0 + j < P.B) dst[(int64_t)(b0 + j) * P.N] = 256.f * (__uint_as_float(v0[j]) + __uint_as_float(v1[j]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_local(dfree0 + db * 8);
    }
  }
  tc_fence_before();
  __syncthreads();
  // the epilogue may be scheduled now: released at the end, not the start, so
  // its blocks land on SMs this grid is leaving (an early release measured
  // slower at 64 sequences with bf16 weights)
  pdl_trigger();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ epilogues
enum EpiKind { EK_QKV = 0, EK_WO = 2, EK_GU = 3, EK_DOWN = 4, EK_PREP_X = 5, EK_PREP_ATT = 6 };

struct TcEpi {
  int32_t kind, N, B, D, Hq, Hkv, hd, dff, NP;
  uint32_t W, parts, G;      // the GEMM's items, CTAs and groups per 128-row tile: which partials a row has
  float eps;
  int64_t pos, s_max;
  const float* part;
  const float* xin32;        // WO: the layer's input residual (fp32) ...
  const uint16_t* xin16;     // ... or bf16; PREP_X: the vector
  const float* vec;          // DOWN: y; PREP_ATT: the attention output
  float* out;                // QKV: q; WO: y; GU: a; DOWN: z
  uint16_t* kc;
  uint16_t* vc;
  const uint16_t* nw;        // RMSNorm weight the limbs are multiplied by (WO: norm2, DOWN: next norm1, PREP_X: norm1)
  uint8_t* xl;               // limb images written (NULL: none)
  const float* rfac_in;      // QKV, GU: RMSNorm factor of the stage's input per sequence (from its GEMM)
  float* ss_out;             // WO, DOWN, PREP_X: of the vector written
  float* resid_out;          // DOWN of the stack's last layer
  uint16_t* out_bf16;
  float rope[64][2];
  const int32_t* posb;       // ragged positions: posb[b] (device copy in the run's parameters) or NULL
  int64_t kv_bstride;        // cache rows from sequence b to b + 1 (0: the rows share one cache)
  const float* rope_b;       // [B][64][2] with posb
  const int32_t* ptab;       // paged caches: slot t of sequence b in page ptab[b * pstride + (t >> pshift)]
  int32_t pshift, pstride;
};

// Position of element k, limb column c of a group's B-operand image.  Inside
// each 16-wide slice the order of k follows the A operand's tensor-memory
// columns: (0,1) (8,9) (2,3) (10,11) (4,5) (12,13) (6,7) (14,15).
__device__ __forceinline__ int64_t limb_offset(int NP, int k, int c) {
  const int kk = k & 63, j = kk >> 4, k16 = kk & 15;
  const int kap = (k16 < 8 ? 4 * (k16 >> 1) + (k16 & 1) : 4 * ((k16 - 8) >> 1) + 2 + (k16 & 1)) + 16 * j;
  return (int64_t)(k >> 6) * NP * 128 + (c >> 3) * SBO + (kap >> 3) * LBO + (c & 7) * 16 + (kap & 7) * 2;
}
// v * 2^-8 as an fp16 high part (column b) and remainder (column B + b).
__device__ __forceinline__ void put_limbs(uint8_t* xl, int NP, int B, int k, int b, float v) {
  const float sv = v * (1.0f / 256.f);
  const __half h0 = __float2half_rn(sv);
  const __half h1 = __float2half_rn(sv - __half2float(h0));
  *reinterpret_cast<__half*>(xl + limb_offset(NP, k, b)) = h0;
  *reinterpret_cast<__half*>(xl + limb_offset(NP, k, B + b)) = h1;
}

__global__ void __launch_bounds__(256, 2) tc_epi_kernel(const __grid_constant__ TcEpi E) {
  constexpr int U = TC_MAX_B / 16;  // sequences a warp takes in one pass: w + 8 u, then w + 8 (u + U)
  __shared__ float rfac[TC_MAX_B];
  const int tid = threadIdx.x, B = E.B, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();  // the previous kernel's outputs (partials, sums of squares, vectors)
  if (E.rfac_in && tid < B) rfac[tid] = __ldcg(E.rfac_in + tid);  // RMSNorm factor of the stage input
  __syncthreads();
  const bool two = E.kind == EK_QKV || E.kind == EK_GU;  // an item is two packed rows, 16T + gg and + 8
  const int64_t items = two ? (int64_t)(E.N / 16) * 8 : E.N;
  const int64_t i0 = items * blockIdx.x / gridDim.x, i1 = items * (blockIdx.x + 1) / gridDim.x;
  // Warp w takes sequences w, w + 8, ...; its lanes take the CTA's items, so
  // that the partials, the [B][N] vectors and the limb images are read and
  // written along rows (coalesced).  For an item a lane first loads what all
  // its sequences need (the split-K partials slot by slot, each sum in CTA
  // order, then the vectors), so that those loads are in flight together,
  // and then computes and stores sequence by sequence.
#pragma unroll 1
  for (int bh = warp; bh < B; bh += 8 * U) {  // (one pass when B <= 8 U)
    float ss[U];
#pragma unroll
    for (int u = 0; u < U; ++u) ss[u] = 0.f;
    for (int64_t it = i0 + lane; it < i1; it += 32) {
      const int i = (int)it;
      const int row0 = two ? 16 * (i >> 3) + (i & 7) : i;  // (row0 + 8 lies in the same 128-row tile)
      float p0[U], p1[U], xv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) p0[u] = p1[u] = xv[u] = 0.f;
      if (E.kind != EK_PREP_X && E.kind != EK_PREP_ATT) {
        const uint32_t r = (uint32_t)row0 >> 7;
        const int ns = (int)(owner32(E.W, E.parts, (r + 1) * E.G - 1) - owner32(E.W, E.parts, r * E.G)) + 1;
        // four slots at a time: their loads are issued together, then added
        // in slot order
        for (int s0 = 0; s0 < ns; s0 += 4) {
          float l0[4][U], l1[4][U];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float* ps = E.part + (int64_t)(s0 + j) * B * E.N + row0;
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int b = bh + 8 * u;
              const bool ok = s0 + j < ns && b < B;
              l0[j][u] = ok ? __ldcg(ps + (int64_t)b * E.N) : 0.f;
              l1[j][u] = ok && two ? __ldcg(ps + (int64_t)b * E.N + 8) : 0.f;
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int u = 0; u < U; ++u)
              if (s0 + j < ns) {
                p0[u] += l0[j][u];
                p1[u] += l1[j][u];
              }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {  // the vector the stage adds to (WO, DOWN) or converts (PREP)
        const int b = bh + 8 * u;
        if (b >= B) continue;
        const int64_t o = (int64_t)b * E.D + i;
        if (E.kind == EK_WO || E.kind == EK_PREP_X)
          xv[u] = E.xin32 ? __ldcg(E.xin32 + o) : bf16_bits_to_f32(E.xin16[o]);
        else if (E.kind == EK_DOWN)
          xv[u] = __ldcg(E.vec + o);
        else if (E.kind == EK_PREP_ATT)
          xv[u] = __ldcg(E.vec + (int64_t)b * E.N + i);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int b = bh + 8 * u;
        if (b >= B) continue;
        switch (E.kind) {
          case EK_QKV: {
            const int T = i >> 3, gg = i & 7, tph = E.hd / 16, head = T / tph, ii = 8 * (T % tph) + gg;
            const float r = rfac[b];
            float v0 = p0[u] * r, v1 = p1[u] * r;
            if (head < E.Hq + E.Hkv) {  // RoPE on q and k: pair (ii, ii + hd/2)
              const float c = E.rope_b ? E.rope_b[((int64_t)b * 64 + ii) * 2] : E.rope[ii][0];
              const float sn = E.rope_b ? E.rope_b[((int64_t)b * 64 + ii) * 2 + 1] : E.rope[ii][1];
              const float x0 = v0, x1 = v1;
              v0 = x0 * c - x1 * sn;
              v1 = x0 * sn + x1 * c;
            }
            if (head < E.Hq) {
              float* qp = E.out + (int64_t)b * E.Hq * E.hd + (int64_t)head * E.hd;
              qp[ii] = v0;
              qp[ii + E.hd / 2] = v1;
            } else {
              const bool is_k = head < E.Hq + E.Hkv;
              const int kvh = is_k ? head - E.Hq : head - E.Hq - E.Hkv;
              const int64_t pb = E.posb ? (int64_t)E.posb[b] : E.pos;
              int64_t rr = (int64_t)b * E.kv_bstride + (int64_t)kvh * E.s_max + pb;
              if (E.pshift) {  // the row inside the page that holds slot pb
                const int64_t pg = E.ptab[(int64_t)b * E.pstride + (pb >> E.pshift)];
                rr = ((pg * E.Hkv + kvh) << E.pshift) + (pb & ((1ll << E.pshift) - 1));
              }
              uint16_t* row = (is_k ? E.kc : E.vc) + rr * E.hd;
              row[ii] = f32_to_bf16_bits(v0);
              row[ii + E.hd / 2] = f32_to_bf16_bits(v1);
            }
            break;
          }
          case EK_GU: {
            const int j = 8 * (i >> 3) + (i & 7);
            const float r = rfac[b], gt = p0[u] * r, up = p1[u] * r;
            const float av = gt / (1.0f + expf(-gt)) * up;
            E.out[(int64_t)b * E.dff + j] = av;
            if (E.xl) put_limbs(E.xl, E.NP, B, j, b, av);
            break;
          }
          case EK_WO: {
            const int64_t o = (int64_t)b * E.D + i;
            const float y = xv[u] + p0[u];
            E.out[o] = y;
            ss[u] = fmaf(y, y, ss[u]);
            if (E.xl) put_limbs(E.xl, E.NP, B, i, b, y * bf16_bits_to_f32(E.nw[i]));
            break;
          }
          case EK_DOWN: {
            const int64_t o = (int64_t)b * E.D + i;
            const float z = xv[u] + p0[u];
            E.out[o] = z;
            ss[u] = fmaf(z, z, ss[u]);
            if (E.xl) put_limbs(E.xl, E.NP, B, i, b, z * bf16_bits_to_f32(E.nw[i]));
            if (E.resid_out) E.resid_out[o] = z;
            if (E.out_bf16) E.out_bf16[o] = f32_to_bf16_bits(z);
            break;
          }
          case EK_PREP_X: {
            const float x = xv[u];
            ss[u] = fmaf(x, x, ss[u]);
            put_limbs(E.xl, E.NP, B, i, b, x * bf16_bits_to_f32(E.nw[i]));
            break;
          }
          default:  // EK_PREP_ATT: the attention output, no norm
            put_limbs(E.xl, E.NP, B, i, b, xv[u]);
            break;
        }
      }
    }
    if (E.ss_out) {  // this CTA's sum of squares of each sequence: the lanes' sums in a fixed tree
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int b = bh + 8 * u;
        if (b >= B) continue;
        float v = ss[u];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) E.ss_out[blockIdx.x * B + b] = v;
      }
    }
  }
}

// ------------------------------------------------------------------ host
int g_tc_ready[64] = {0};

int prepare(int wtype) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= 64) return DDL_ERR_UNSUPPORTED;
  const int bit = wtype == DDL_W_INT4 ? 1 : 2;
  if (g_tc_ready[dev] & bit) return DDL_OK;
  e = cudaFuncSetAttribute(wtype == DDL_W_INT4 ? (const void*)tc_gemm_kernel<DDL_W_INT4>
                                               : (const void*)tc_gemm_kernel<DDL_W_BF16>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e != cudaSuccess) return cuda_status(e);
  g_tc_ready[dev] |= bit;
  return DDL_OK;
}

int64_t al256(int64_t x) { return (x + 255) & ~int64_t(255); }
uint32_t al1024(uint32_t x) { return (x + 1023u) & ~1023u; }

// The GEMM's CTAs for matrix m on C SMs (each holds an equal share of the
// NR * G items; every CTA at least one) and the most partials a tile gets.
void split_of(const MatGeom& m, int C, uint32_t& parts, int& slots) {
  const uint32_t NR = (uint32_t)(m.NT + 7) / 8, W = NR * (uint32_t)m.G;
  parts = W < (uint32_t)C ? W : (uint32_t)C;
  for (;; --parts) {  // a tile's partials within TC_MAX_SPLIT (a no-op at the model shapes)
    slots = 0;
    for (uint32_t r = 0; r < NR; ++r) {
      const int n = (int)(owner32(W, parts, (r + 1) * m.G - 1) - owner32(W, parts, r * m.G)) + 1;
      if (n > slots) slots = n;
    }
    if (slots <= TC_MAX_SPLIT || parts == 1) return;
  }
}

void tc_sizes(const ddl_shape& s, int B, int C, int64_t& part_floats, int64_t& xl_bytes) {
  MatGeom mg[4];
  make_geoms(s, DDL_W_INT4, mg);
  part_floats = 0;
  xl_bytes = 0;
  for (int k = 0; k < 4; ++k) {
    uint32_t parts;
    int slots;
    split_of(mg[k], C, parts, slots);
    const int64_t p = (int64_t)slots * mg[k].N * B;
    if (p > part_floats) part_floats = p;
    const int64_t x = (int64_t)mg[k].G * tc_ncols(B) * 128;
    if (x > xl_bytes) xl_bytes = x;
  }
}

int launch_epi(const TcEpi& E, cudaStream_t cs) {
  void* args[] = {const_cast<TcEpi*>(&E)};
  return cuda_status(launch_pdl((const void*)tc_epi_kernel, dim3(TC_EPI_CTAS), dim3(256), args, 0, cs));
}

TcEpi epi_base(const TcRun& R) {
  TcEpi E;
  memset(&E, 0, sizeof E);
  E.B = R.B;
  E.D = R.D;
  E.Hq = R.Hq;
  E.Hkv = R.Hkv;
  E.hd = R.hd;
  E.dff = R.dff;
  E.NP = tc_ncols(R.B);
  E.eps = R.eps;
  E.pos = R.pos;
  E.s_max = R.s_max;
  E.part = R.part;
  memcpy(E.rope, R.rope, sizeof E.rope);
  E.posb = R.posb;
  E.kv_bstride = R.kv_bstride;
  E.rope_b = R.rope_b;
  E.ptab = R.ptab;
  E.pshift = R.pshift;
  E.pstride = R.pstride;
  return E;
}

}  // namespace

int64_t tc_workspace_bytes(const ddl_shape& s, int B, int wtype) {
  (void)wtype;
  int dev = 0, C = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&C, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  int64_t pf, xb;
  tc_sizes(s, B, C, pf, xb);
  return al256(pf * 4) + al256(xb) + al256((int64_t)2 * TC_EPI_CTAS * B * 4) + al256((int64_t)2 * B * 4);
}

void tc_workspace_carve(const ddl_shape& s, int B, int wtype, uint8_t* base, TcRun& R) {
  (void)wtype;
  int64_t pf, xb;
  tc_sizes(s, B, R.C, pf, xb);
  R.part = reinterpret_cast<float*>(base);
  R.xl = base + al256(pf * 4);
  R.ss = reinterpret_cast<float*>(R.xl + al256(xb));
  R.rfac = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(R.ss) + al256((int64_t)2 * TC_EPI_CTAS * B * 4));
}

int tc_begin(const TcRun& R, void* stream) {
  cudaStream_t cs = (cudaStream_t)stream;
  int st = prepare(R.wtype);
  if (st) return st;
  int64_t pf, xb;
  ddl_shape sh;
  sh.D = R.D; sh.H_q = R.Hq; sh.H_kv = R.Hkv; sh.head_dim = R.hd; sh.d_ff = R.dff; sh.eps = R.eps; sh.rope_base = 1.0;
  tc_sizes(sh, R.B, R.C, pf, xb);
  cudaError_t e = cudaMemsetAsync(R.xl, 0, (size_t)xb, cs);  // padding columns stay zero
  if (e != cudaSuccess) return cuda_status(e);
  // the first layer's QKV operands and the sums of squares of its input
  TcEpi E = epi_base(R);
  E.kind = EK_PREP_X;
  E.N = R.D;
  if (R.l0 == 0) {
    E.xin32 = R.resid_in;
    E.xin16 = R.resid_in ? nullptr : R.x_bf16;
  } else {
    E.xin32 = R.Z + (int64_t)((R.l0 - 1) & 1) * R.B * R.D;
  }
  E.nw = R.layers[0].norm1;
  E.xl = R.xl;
  E.ss_out = R.ss;
  return launch_epi(E, cs);
}

int tc_stage(const TcRun& R, int layer, int st, void* stream) {
  cudaStream_t cs = (cudaStream_t)stream;
  const int gl = R.l0 + layer, B = R.B, NP = tc_ncols(B);
  const TcLayer& Ly = R.layers[layer];
  int rc;
  if (st == ST_WO) {  // the attention output becomes the Wo operands
    TcEpi E = epi_base(R);
    E.kind = EK_PREP_ATT;
    E.N = R.Hq * R.hd;
    E.vec = R.attn;
    E.xl = R.xl;
    if ((rc = launch_epi(E, cs))) return rc;
  }
  const MatGeom& m = R.mg[stage_mat(st)];
  TcGemm G;
  memset(&G, 0, sizeof G);
  G.N = m.N;
  G.NT = m.NT;
  G.G = m.G;
  G.Sk = m.Sk;
  G.Gc = m.Gc;
  G.glast = m.G - (m.Sk - 1) * m.Gc;
  G.NR = (m.NT + 7) / 8;
  if ((uint64_t)G.NR * (uint64_t)m.G * (uint64_t)R.C >= (1ull << 32)) return DDL_ERR_UNSUPPORTED;  // owner32
  int slots;
  split_of(m, R.C, G.parts, slots);
  G.W = (uint32_t)G.NR * (uint32_t)m.G;
  G.NP = NP;
  G.B = B;
  const uint32_t BB = R.wtype == DDL_W_INT4 ? QBLK_BYTES : BF16_BLK_BYTES;
  // groups per stage: as many as keep three stages within 200 KB (at most 8)
  G.gs = 8;
  while (G.gs > 1 && 3 * (al1024(8 * BB * G.gs) + al1024((uint32_t)NP * 128 * G.gs)) > 200u * 1024u) --G.gs;
  // four A buffers (a deeper A ring measured slower), then accumulators of
  // NP columns plus 16 of headroom (the read-out loads 16 columns at a time,
  // up to column 2B + 14): two when they fit, else one
  G.dstride = NP + 16;
  G.na = 4;
  G.nd = G.na * A_COLS + 2 * G.dstride <= TMEM_COLS ? 2 : 1;
  G.wbytes = al1024(8 * BB * G.gs);
  G.stage_bytes = G.wbytes + al1024((uint32_t)NP * 128 * G.gs);
  G.w = Ly.packed + m.woff;
  G.xl = R.xl;
  G.part = R.part;
  if (st == ST_QKV || st == ST_GU) {  // this GEMM also reduces its epilogue's RMSNorm factors
    G.ss_in = R.ss + (st == ST_GU ? TC_EPI_CTAS * B : 0);
    G.rfac = R.rfac + (st == ST_GU ? B : 0);
    G.ss_K = R.D;
    G.eps = R.eps;
  }
  G.status = R.status;
  G.wait_ns = R.wait_ns;
  // as many ring stages as fit (at most MAX_STAGES); at least half of an SM's
  // shared memory, so that no two CTAs share an SM and its 512 tensor-memory
  // columns
  G.stages = (int32_t)((200u * 1024u) / G.stage_bytes);
  if (G.stages > MAX_STAGES) G.stages = MAX_STAGES;
  if (G.stages < 2) return DDL_ERR_UNSUPPORTED;
  size_t smem = (size_t)G.stages * G.stage_bytes + 1024;
  if (smem < 116 * 1024) smem = 116 * 1024;
  if (smem > 227 * 1024) return DDL_ERR_UNSUPPORTED;
  {
    void* args[] = {&G};
    const int grid = (int)G.parts;
    const void* fn = R.wtype == DDL_W_INT4 ? (const void*)tc_gemm_kernel<DDL_W_INT4> : (const void*)tc_gemm_kernel<DDL_W_BF16>;
    if ((rc = cuda_status(launch_pdl(fn, dim3(grid), dim3(GT), args, smem, cs)))) return rc;
  }
  TcEpi E = epi_base(R);
  E.kind = st;
  E.N = m.N;
  E.W = G.W;
  E.parts = G.parts;
  E.G = (uint32_t)m.G;
  switch (st) {
    case ST_QKV:
      E.out = R.q;
      E.kc = Ly.kc;
      E.vc = Ly.vc;
      E.rfac_in = R.rfac;
      break;
    case ST_WO:
      if (gl == 0) {
        E.xin32 = R.resid_in;
        E.xin16 = R.resid_in ? nullptr : R.x_bf16;
      } else {
        E.xin32 = R.Z + (int64_t)((gl - 1) & 1) * B * R.D;
      }
      E.out = R.y;
      E.nw = Ly.norm2;
      E.xl = R.xl;
      E.ss_out = R.ss + TC_EPI_CTAS * B;
      break;
    case ST_GU:
      E.out = R.a;
      E.xl = R.xl;
      E.rfac_in = R.rfac + B;
      break;
    default: {  // ST_DOWN
      E.vec = R.y;
      E.out = R.Z + (int64_t)(gl & 1) * B * R.D;
      if (layer + 1 < R.L) {  // the next layer's QKV operands
        E.nw = R.layers[layer + 1].norm1;
        E.xl = R.xl;
        E.ss_out = R.ss;
      }
      if (R.final_last && layer == R.L - 1) {
        E.resid_out = R.resid_out;
        E.out_bf16 = R.out_bf16;
      }
      break;
    }
  }
  return launch_epi(E, cs);
}

}  // namespace ddl
