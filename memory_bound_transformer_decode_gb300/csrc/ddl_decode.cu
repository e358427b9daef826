// ddl_decode.cu -- the decode step: one persistent kernel that streams every
// weight and KV byte of an L-layer stack once, and its host runtime.
//
// Per layer the kernel runs five stages (primer "把基础打牢" §1.1 block, §1.2
// decode_step):
//   QKV  : rmsnorm(x) folded into the GEMV (W (x*w1)) * r, INT4 codes expanded
//          in registers and multiplied on the tensor cores, RoPE on q and k,
//          bf16 k and v appended to the cache at slot pos (Unsloth/Qwen-27B
//          article §二.1 fused RMSNorm+RoPE, §二.3 in-register 4-bit expansion)
//   ATT  : split-KV GQA decode attention: each K/V head is read once, in
//          place, for its whole query group (same article §二.2), with an
//          online softmax per 16-key tile (FlashAttention-style tiling, roofline
//          reply §四); the last CTA to finish a sequence merges its
//          split-KV partial softmax states
//   WO   : y = x + attn Wo
//   GU   : rmsnorm(y) folded into the gate/up GEMV, silu(g) * u in the epilogue
//          (Unsloth/Qwen-27B article §二.1 fused SwiGLU)
//   DOWN : z = y + a Wd
// Every consumer warp owns a ring of DEPTH shared-memory slots filled by TMA
// (1-D bulk copies of weight blocks, 2-D tensor copies of K/V tiles).  One
// producer warp keeps all the rings full: its lane w walks consumer warp w's
// work and refills a slot as soon as the consumer hands it back (an "empty"
// mbarrier), running ahead across stage (and layer) boundaries because
// weights and the KV history do not depend on the token being decoded; the
// consumers only wait for data, compute and hand slots back.  Stages are separated by a grid-wide barrier (one
// cooperative launch for the whole stack) or by kernel boundaries (one launch
// per stage).  All waits are bounded: a wait that gives up sets the status
// word in the workspace and the kernel returns.
#include <math.h>
#include <mutex>
#include <stdio.h>
#include <string.h>

#include <unordered_map>
#include <vector>

#include <cudaTypedefs.h>

#include "ddl_device.cuh"
#include "ddl_internal.h"
#include "ddl_tc.h"

namespace ddl {

// ------------------------------------------------------------------ shared memory
// The parameters that are read with a run-time index (per layer, per matrix,
// per RoPE frequency) are copied to shared memory at launch, so that a stage
// start does not wait on constant-cache misses.
struct SParams {
  MatGeom mg[4];
  float rope[64][2];
  LayerDev layers[MAX_LAYERS];
};
extern __shared__ __align__(1024) uint8_t g_smem[];
constexpr int SM_RING = 0;
constexpr int SM_RING_BYTES = NW * DEPTH * SLOT_BYTES;
constexpr int SM_BARS = SM_RING_BYTES;                // "full" barriers: a slot's copy landed
constexpr int SM_EBARS = SM_BARS + NW * DEPTH * 8;    // "empty" barriers: the consumer handed a slot back
constexpr int SM_XBAR = SM_EBARS + NW * DEPTH * 8;    // the batch-1 prologue's x copy
constexpr int SM_SCR = SM_BARS + 512;
constexpr int XF_BYTES = XF_CHUNKS * GC * 4 * 2 * 4 * 8;  // x fragments: chunks x batch <= 8
constexpr int SX_BYTES = XF_CHUNKS * GC * NARROW_B * 4;     // per-group sums of x (wide: 2 chunks x 16)
constexpr int SM_SCR_BYTES = 71 * 1024;
constexpr int SM_NW = SM_SCR + SM_SCR_BYTES;               // the panel's norm weights (bf16)
constexpr int SM_NW_BYTES = XF_CHUNKS * GC * DDL_GROUP * 2;
constexpr int SM_MISC = SM_NW + SM_NW_BYTES;
constexpr int SM_MISC_BYTES = 2048;
constexpr int SM_SPAR = SM_MISC + SM_MISC_BYTES;             // copies of the indexed parameters
constexpr int SM_CTX = SM_SPAR + (((int)sizeof(SParams) + 255) & ~255);  // stage context, warp cursors
constexpr int SM_CTX_BYTES = 4096;
constexpr int SM_TOTAL = SM_CTX + SM_CTX_BYTES;
constexpr int XZ_OFF = XF_BYTES + SX_BYTES + NW * 32 * 4;  // zero x fragments for blocks past a slot's end
constexpr int XZ_BYTES = 2048;                             // covers both fragment layouts
static_assert(XZ_OFF + XZ_BYTES <= SM_SCR_BYTES, "x fragments do not fit");
static_assert(SM_XBAR + 8 <= SM_SCR, "barriers");
static_assert(NW * 2 * (MAX_GH * (128 + 2) + 3) * 4 <= SM_SCR_BYTES, "attention records do not fit");
static_assert(SM_TOTAL <= 227 * 1024, "shared memory budget");
static_assert(SM_SPAR % 16 == 0, "parameter copy alignment");
static_assert(sizeof(Params) <= 32000, "kernel parameters (with the K/V tensor maps) exceed the launch limit");
static_assert((SLOT_BYTES % 1024 == 512 && SLOT_BYTES >= 512 + 16 * 128 * 2) ||
                  (SLOT_BYTES % 1024 == 0 && SLOT_BYTES >= 16 * 128 * 2),
              "K/V boxes need 1024-byte boundaries inside 512-byte aligned slots");
__device__ __forceinline__ const SParams& sp() { return *reinterpret_cast<const SParams*>(g_smem + SM_SPAR); }

// Position of sequence b's new token, its 16-key tiles (the last holds the new
// token), and the RoPE (cos, sin) of head-dimension pair i at that position.
__device__ __forceinline__ int64_t seq_pos(const Params& P, int b) { return P.ragged ? P.posb[b] : P.pos; }
__device__ __forceinline__ int att_tiles(const Params& P, int64_t seq) {
  return P.ragged ? (int)(P.posb[seq / P.Hkv] / 16) + 1 : P.nt_att;
}
// First cache-view row of attention sequence seq = (b, kv head) (per-sequence
// positions and prefill, whose rows may share one cache).
__device__ __forceinline__ int64_t att_row0(const Params& P, int64_t seq) {
  return (seq / P.Hkv) * P.kv_bstride + (seq % P.Hkv) * P.s_max;
}
// Cache-view row of slot t of attention sequence seq = (b, kv head): in a
// paged cache the row inside the page that holds slot t (the page table is
// read-only for the whole call).
__device__ __forceinline__ int64_t att_row(const Params& P, int64_t seq, int64_t t) {
  if (P.pshift) {
    const int64_t b = seq / P.Hkv, kvh = seq % P.Hkv;
    const int64_t pg = __ldg(P.ptab + b * P.pstride + (t >> P.pshift));
    return ((pg * P.Hkv + kvh) << P.pshift) + (t & ((1ll << P.pshift) - 1));
  }
  return att_row0(P, seq) + t;
}
__device__ __forceinline__ float2 rope_cs(const Params& P, int b, int i) {
  if (P.ragged) return *reinterpret_cast<const float2*>(P.rope_b + ((int64_t)b * 64 + i) * 2);
  return make_float2(sp().rope[i][0], sp().rope[i][1]);
}

// An empty partial slot word: two all-ones NaNs, a pattern that fp32
// arithmetic does not produce (its NaN results are canonical).
constexpr uint64_t PART_EMPTY = ~0ull;

struct Misc {
  float rnorm[MAX_B];
  float escale[MAX_B];     // 2^e of the staged x of each sequence
  float edown[MAX_B];      // 2^-e
  float red[NW][2 * MAX_B];
  int kc_lo, nkc;
  int abort;
  int seg_n[NW];
  long long seg_first[NW], seg_last[NW];
  long long mseq[8];       // sequences this CTA merges last
  uint32_t xuse;           // batch-1 prologue copies completed on the x barrier so far (its phase)
  int nruns;               // CTA merge: runs of warp records of one sequence
  int run_first[2 * NW];
  uint32_t run_vmask[2 * NW];
  long long run_seq[2 * NW], run_out[2 * NW];
  uint32_t cmax[MAX_B];    // running max |output * consumer norm weight| of this stage (float bits)
};
static_assert(sizeof(Misc) <= SM_MISC_BYTES, "misc");

enum SlotKind { SK_GEMV = 0, SK_K = 1, SK_V = 2 };

struct SlotDesc {
  int kind, cnt;
  uint32_t a;  // GEMV: stream block index; K/V: first row of the tile in the [rows][hd] cache view
};
// Producer cursor over one consumer warp's slots of every stage of the
// launch (held by the producer lane serving that warp); it caches the current
// stage's stream bases so that issuing a slot reads no per-layer parameter
// with a run-time index.
struct Cursor {
  int s, st;              // flattened stage and its kind
  uint32_t pos, end;      // work index and end: GEMV panel blocks, ATT 2 x tiles (K, V)
  uint32_t a;             // GEMV: stream block index of pos; ATT: cache-view row of the tile
  int aseq, ai;           // ATT: sequence and tile index of the tile
  const uint8_t* wbase;   // GEMV: block stream of the matrix (INT4: codes and scales)
  const void* kmap;       // ATT: tensor maps of the layer's caches
  const void* vmap;
  int kc, T, gi, gk;      // GEMV: (k-chunk, tile, group) of work index `pos`
  int NT, Sk, Gc, G;      // GEMV: geometry of the matrix
  int pk0, pk1;           // GEMV: k-chunks of this CTA's panel
};
// A consumer warp's view of its ring: the next slot to consume sits at
// slot(), lands on full barrier bar() with phase parity `phase`, and is
// handed back on empty barrier ebar(); advance() steps to the slot after it.
struct Ring {
  uint32_t slot0, bar0, ebar0;
  uint32_t idx, phase;
  __device__ __forceinline__ uint32_t slot() const { return slot0 + idx * SLOT_BYTES; }
  __device__ __forceinline__ uint32_t bar() const { return bar0 + idx * 8; }
  __device__ __forceinline__ uint32_t ebar() const { return ebar0 + idx * 8; }
  __device__ __forceinline__ void advance() {
    if (++idx == DEPTH) {
      idx = 0;
      phase ^= 1u;
    }
  }
  __device__ __forceinline__ Ring next() const {
    Ring r = *this;
    r.advance();
    return r;
  }
};

// Per-stage constants of a GEMV stage, read once from the parameters.
struct GemvCtx {
  MatGeom m;
  int st, layer, gl;
  const float* xin32;     // layer input (fp32) or NULL
  const uint16_t* xin16;  // layer input (bf16) when xin32 is NULL (QKV / WO of layer 0)
  uint16_t* kc;           // K, V caches (QKV epilogue)
  uint16_t* vc;
  float* zout;            // residual output of this layer (DOWN)
  bool final_layer;
  int p, cl;              // this CTA's panel and its index among the panel's CTAs
};

// CTA-wide state in shared memory, so that nothing lives in local memory:
// the current weight stage's context and each consumer warp's ring between
// stages.
// A warp's place in each stage kind, the same for every layer of a launch:
// computed once at launch so that entering a stage costs no divisions.
struct Entry {
  uint32_t lo, hi;           // work range: GEMV panel work indices, ATT 16-key tiles
  int32_t T, kc, gi, gk;     // GEMV: (tile, k-chunk, group) at lo and the chunk's groups
  int16_t p, cl, pk0, pk1;   // GEMV: panel, CTA index in the panel, the panel's k-chunks
  uint32_t first;            // GEMV: panel-local index of the first warp holding tile T in this panel
  uint32_t omask[2];         // GEMV: partial slots (bit p J + j) of the first two tiles this warp owns
};
// This CTA's part of the attention stage, the same for every layer of a
// launch: its range of (sequence, 16-key tile) work and, per sequence it
// touches, the first CTA holding a tile of it and how many CTAs do.
struct AttCta {
  int32_t clo, chi;  // tiles [clo, chi) of the B * H_kv * nt work order
  int32_t s0, ns;    // sequences s0 .. s0 + ns - 1 (ns <= 8, checked by the host)
  int32_t cf[8];
  int32_t span[8];  // CTAs cf .. cf + span - 1 (with fewer tiles than CTAs some hold none)
  uint32_t n[8];    // the CTAs that hold a tile of it: arrivals before its merge
};
struct Ctx {
  GemvCtx E;
  AttCta att;
  Ring ring[NW];
  Entry ent[NW][NSTAGE];
};
static_assert(sizeof(Ctx) <= SM_CTX_BYTES, "context");
__device__ __forceinline__ Ctx& ctx() { return *reinterpret_cast<Ctx*>(g_smem + SM_CTX); }

// ------------------------------------------------------------------ work split
__device__ __forceinline__ void att_range(const Params& P, int64_t& lo, int64_t& hi) {
  const int64_t Ta = (int64_t)P.B * P.Hkv * P.nt_att, C = gridDim.x;
  const int64_t clo = range_lo(Ta, C, blockIdx.x), chi = range_lo(Ta, C, blockIdx.x + 1);
  const int w = threadIdx.x >> 5;
  lo = clo + range_lo(chi - clo, NW, w);
  hi = clo + range_lo(chi - clo, NW, w + 1);
}
// Partial slots of split tile T (bit p J + j: the j-th warp holding blocks of
// T in panel p), read by the tile's owner.
__device__ __noinline__ uint32_t owned_slots(const MatGeom& m, int T) {  // bit f = p * J + j
  uint32_t mask = 0;
  for (int p = 0; p < m.NP; ++p) {
    const uint32_t Gp = panel_groups(m, p);
    const uint32_t v0 = work_owner(m, p, (uint32_t)T * Gp, NW), v1 = work_owner(m, p, (uint32_t)(T + 1) * Gp - 1, NW);
    for (uint32_t v = v0; v <= v1; ++v)
      if (!warp_empty(m, p, v, NW)) mask |= 1u << (p * m.J + (v - v0));
  }
  return mask;
}
// Compute this warp's entry for every stage kind the launch runs (once per
// launch; a launch of the attention stage alone, as the tensor-core path
// makes one per layer, skips the weight stages' entries, which cost up to
// tens of microseconds on some CTAs).
__device__ __noinline__ void compute_entries(const Params& P) {
  const int warp = threadIdx.x >> 5;
  uint32_t kinds = 0;
  for (int s = P.stage_begin; s < P.stage_end && kinds != (1u << NSTAGE) - 1; ++s) kinds |= 1u << (s % NSTAGE);
  for (int st = 0; st < NSTAGE; ++st) {
    if (!(kinds & (1u << st))) continue;
    Entry e;
    if (st == ST_ATT) {
      int64_t lo, hi;
      att_range(P, lo, hi);
      e.lo = (uint32_t)lo;
      e.hi = (uint32_t)hi;
      e.T = e.kc = e.gi = e.gk = 0;
      e.p = e.cl = e.pk0 = e.pk1 = 0;
    } else {
      const MatGeom& m = sp().mg[stage_mat(st)];
      const int p = panel_of_cta(m, blockIdx.x);
      uint32_t lo, hi;
      warp_work(m, p, blockIdx.x - m.pc[p], warp, NW, lo, hi);
      e.lo = lo;
      e.hi = hi;
      e.p = (int16_t)p;
      e.cl = (int16_t)(blockIdx.x - m.pc[p]);
      e.pk0 = m.pk[p];
      e.pk1 = m.pk[p + 1];
      e.T = e.kc = e.gi = 0;
      e.gk = 1;
      e.first = 0;
      e.omask[0] = e.omask[1] = 0u;
      if (lo < hi) {
        int T, kc, gi;
        work_coord(m, p, lo, T, kc, gi);
        e.T = T;
        e.kc = kc;
        e.gi = gi;
        e.gk = chunk_groups(m, kc);
        const uint32_t Gp = panel_groups(m, p);
        e.first = work_owner(m, p, (uint32_t)T * Gp, NW);  // later tiles of the range start in it
        if (p == 0) {  // owned: split tiles whose first panel-0 block is in the range
          uint32_t mk[2] = {0u, 0u};
          for (uint32_t t = (lo + Gp - 1) / Gp; t * Gp < hi && mk[1] == 0u; ++t)
            if (m.NP > 1 || (t + 1) * Gp > hi) {
              const uint32_t k = owned_slots(m, (int)t);
              if (mk[0] == 0u) mk[0] = k;
              else mk[1] = k;
            }
          e.omask[0] = mk[0];
          e.omask[1] = mk[1];
        }
      }
    }
    if ((threadIdx.x & 31) == 0 && warp < NW) ctx().ent[warp][st] = e;
  }
  AttCta& A = ctx().att;
  const int64_t Ta = (int64_t)P.B * P.Hkv * P.nt_att, C = gridDim.x, nt = P.nt_att;
  const int64_t clo = range_lo(Ta, C, blockIdx.x), chi = range_lo(Ta, C, blockIdx.x + 1);
  const int64_t s0 = clo / nt, ns = clo < chi ? (chi - 1) / nt - s0 + 1 : 0;
  if (threadIdx.x == 0) {
    A.clo = (int32_t)clo;
    A.chi = (int32_t)chi;
    A.s0 = (int32_t)s0;
    A.ns = (int32_t)ns;
  }
  if (threadIdx.x < ns && threadIdx.x < 8) {
    const int64_t sq = s0 + threadIdx.x;
    const int64_t cf = owner_of(Ta, C, sq * nt), cl = owner_of(Ta, C, sq * nt + nt - 1);
    A.cf[threadIdx.x] = (int32_t)cf;
    A.span[threadIdx.x] = (int32_t)(cl - cf + 1);
    A.n[threadIdx.x] = (uint32_t)(Ta >= C ? cl - cf + 1 : nt);
  }
}
// RAG: sequences at their own positions (a separate kernel instance, so that
// the shared-position step carries none of its code).
template <int WT, bool RAG>
__device__ __forceinline__ void cursor_enter(const Params& P, Cursor& c, int w) {
  const int st = c.s % NSTAGE;
  c.st = st;
  const LayerDev& Ld = sp().layers[c.s / NSTAGE];
  const Entry& e = ctx().ent[w][st];
  c.pos = e.lo;
  c.end = e.hi;
  if (st == ST_ATT) {
    c.aseq = (int)(e.lo / (uint32_t)P.nt_att);
    c.ai = (int)(e.lo - (uint32_t)c.aseq * (uint32_t)P.nt_att);
    c.pos *= 2;
    c.end *= 2;
    if (RAG && c.ai >= att_tiles(P, c.aseq)) {  // the range starts past a sequence's new token
      c.pos += 2u * (uint32_t)(P.nt_att - c.ai);
      c.ai = 0;
      ++c.aseq;
    }
    // (a range that ends with the sequence it skipped to holds no tile of it:
    // its row is never used, and the page table is not read for it)
    c.a = RAG ? (c.pos < c.end ? (uint32_t)att_row(P, c.aseq, 16 * (int64_t)c.ai) : 0u)
              : (uint32_t)((int64_t)c.aseq * P.s_max + 16 * c.ai);
    c.kmap = &P.kmap[c.s / NSTAGE];
    c.vmap = &P.vmap[c.s / NSTAGE];
  } else {
    const MatGeom& m = sp().mg[stage_mat(st)];
    c.wbase = Ld.packed + m.woff;
    c.NT = m.NT;
    c.Sk = m.Sk;
    c.Gc = m.Gc;
    c.G = m.G;
    c.pk0 = e.pk0;
    c.pk1 = e.pk1;
    c.T = e.T;
    c.kc = e.kc;
    c.gi = e.gi;
    c.gk = e.gk;
    c.a = (uint32_t)c.kc * (uint32_t)c.NT * (uint32_t)c.Gc + (uint32_t)c.T * (uint32_t)c.gk + (uint32_t)c.gi;
  }
}
template <int WT, bool RAG>
__device__ __forceinline__ bool cursor_next(const Params& P, Cursor& c, int w, SlotDesc& d) {
  while (c.pos >= c.end) {
    if (++c.s >= P.stage_end) return false;
    cursor_enter<WT, RAG>(P, c, w);
  }
  if (c.st == ST_ATT) {  // K then V of one 16-key tile
    d.kind = (c.pos & 1) ? SK_V : SK_K;
    d.a = c.a;
    d.cnt = 16;
    if (c.pos & 1) {  // the next tile
      // (sequences at their own positions: tiles past a sequence's new token
      // hold no keys, and the consumer skips them too)
      if (++c.ai == P.nt_att || (RAG && c.ai >= att_tiles(P, c.aseq))) {
        c.pos += 2u * (uint32_t)(P.nt_att - c.ai);
        c.ai = 0;
        ++c.aseq;
        c.a = RAG ? (c.pos + 1 < c.end ? (uint32_t)att_row(P, c.aseq, 0) : 0u) : (uint32_t)((int64_t)c.aseq * P.s_max);
      } else if (RAG && P.pshift && ((16 * c.ai) & ((1 << P.pshift) - 1)) == 0) {
        c.a = (uint32_t)att_row(P, c.aseq, 16 * (int64_t)c.ai);  // the next page
      } else {
        c.a += 16;
      }
    }
    c.pos += 1;
  } else {  // up to PER blocks of one (k-chunk, tile) unit, in panel work order
    constexpr int PER = WT == DDL_W_INT4 ? BLKS_PER_SLOT : BF16_BLKS_PER_SLOT;
    d.kind = SK_GEMV;
    const uint32_t left = c.end - c.pos;
    int n = left < (uint32_t)PER ? (int)left : PER;
    if (n > c.gk - c.gi) n = c.gk - c.gi;
    d.a = c.a;
    d.cnt = n;
    c.pos += n;
    c.gi += n;
    c.a += n;
    if (c.gi == c.gk) {
      c.gi = 0;
      if (++c.kc == c.pk1) {
        c.kc = c.pk0;
        ++c.T;
      }
      c.gk = c.kc == c.Sk - 1 ? c.G - (c.Sk - 1) * c.Gc : c.Gc;
      c.a = (uint32_t)c.kc * (uint32_t)c.NT * (uint32_t)c.Gc + (uint32_t)c.T * (uint32_t)c.gk;
    }
  }
  return true;
}

// A K/V slot holds 16 rows of hd bf16 as hd/64 boxes of 16 rows x 128 bytes
// with the 128-byte swizzle, which wants each box at a 1024-byte boundary:
// ring slots are 512-byte aligned, and one that starts 512 bytes past a
// boundary puts its boxes 512 bytes in (4608-byte slots: they end at its end).
__device__ __forceinline__ uint32_t kv_base(uint32_t slot) { return (slot + 1023u) & ~1023u; }
// Shared address of 16-byte chunk `ch` (head dims 8ch..8ch+7) of row r: half
// ch/8 of the row in its own 2 KB box, chunk ch%8 XOR-ed with row%8.
__device__ __forceinline__ uint32_t kv_addr(uint32_t slot, int r, int ch) {
  return kv_base(slot) + (ch >> 3) * 2048 + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
}
// Issue one slot's copies (by one producer lane).
template <int HD, int WT>
__device__ __forceinline__ void issue_slot(const Cursor& c, const SlotDesc& d, uint32_t slot, uint32_t bar,
                                           uint64_t policy) {
  if (d.kind == SK_GEMV) {
    constexpr bool q4 = WT == DDL_W_INT4;
    constexpr uint32_t BB = q4 ? QBLK_BYTES : BF16_BLK_BYTES;  // INT4: codes and scales together
    const uint32_t wb = d.cnt * BB;
    mbar_arrive_expect_tx(bar, wb);
    bulk_g2s_evict_first(slot, c.wbase + (uint64_t)d.a * BB, wb, bar, policy);
  } else {  // 16 rows of K or V: HD/64 boxes of 16 rows x 128 bytes, swizzled (kv_addr)
    mbar_arrive_expect_tx(bar, 16 * HD * 2);
#pragma unroll
    for (int b = 0; b < HD / 64; ++b)
      tensor2d_g2s(kv_base(slot) + b * 2048, d.kind == SK_K ? c.kmap : c.vmap, b * 64, (int)d.a, bar, policy);
  }
}

// Hand the slot just consumed back to the producer.  The warp's reads of it
// are ordered before the arrival by the warp barrier and the arrival's
// release; a warp that wrote into the slot fenced those writes for the async
// proxy first.
__device__ __forceinline__ void ring_advance(Ring& R, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(R.ebar());
  R.advance();
}

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) { return __uint_as_float(lds32(a)); }
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ float4 bf16x4_f32(uint2 u) {
  return make_float4(bf16lo_f32(u.x), bf16hi_f32(u.x), bf16lo_f32(u.y), bf16hi_f32(u.y));
}

// Optional trace per (stage, CTA): word 0 is %globaltimer at the stage start
// (comparable across SMs), word 15 %clock64 at the same moment, and words
// 1..14 %clock64 at later events (end of the prologue, end of each warp's
// stream, end of the stage, prologue steps), so that intervals within a CTA
// are exact to a cycle; words 16 + w and 24 + w hold the cycles consumer warp
// w spent waiting for its ring's data and the slots it consumed.
__device__ __forceinline__ void trace_ring(const Params& P, int s, uint64_t wait_cycles, uint32_t slots) {
  if (P.trace && (threadIdx.x & 31) == 0) {
    uint64_t* w = P.trace + ((int64_t)(s - P.stage_begin) * gridDim.x + blockIdx.x) * TRACE_WORDS;
    w[16 + (threadIdx.x >> 5)] = wait_cycles;
    w[24 + (threadIdx.x >> 5)] = slots;
  }
}
__device__ __forceinline__ void trace_stamp(const Params& P, int s, int slot) {
  if (P.trace) {
    uint64_t* w = P.trace + ((int64_t)(s - P.stage_begin) * gridDim.x + blockIdx.x) * TRACE_WORDS;
    if (slot == 0) {
      const uint64_t c = clock64();
      w[15] = c;
      w[0] = globaltimer();
    } else {
      w[slot] = clock64();
    }
  }
}



// ------------------------------------------------------------------ grid barrier
// Arrival: the CTA's writes of this stage (ordered before by the block
// barrier) become visible no later than the release.  The wait (acquiring
// polls) orders the next stage's reads after every CTA's arrival; between
// the two the CTA prepares its next stage.
__device__ void grid_arrive(const Params& P) {
  csync();
  if (threadIdx.x == NTHREADS - 32) red_release_gpu_add(P.ctrl, 1u);  // not thread 0: see gemv_prep
}
__device__ __forceinline__ bool grid_wait(const Params& P, uint32_t target, Misc& M) {
  if (threadIdx.x == 0) {
    uint64_t t0 = 0;
    for (uint32_t it = 1; ld_acquire_gpu(P.ctrl) < target; ++it) {
      if ((it & 255u) != 0) continue;
      const uint64_t now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > P.wait_ns) {
        atomicExch(P.ctrl + 1, STATUS_TIMEOUT);
        M.abort = 1;
        break;
      }
    }
  }
  csync();
  return !M.abort;
}

// ------------------------------------------------------------------ GEMV prologue
// Stages this CTA's panel of the activation (k-chunks pk[p]..pk[p+1]-1) as
// m16n8k16 B fragments: column 2b is the fp16 "high" part of sequence b's
// x * norm weight * 2^-8, column 2b+1 the fp16 remainder, so x is carried to
// ~22 significant bits for |x w| >= 32 and to an absolute 2^-17 below (range
// |x w| < 2^24 with no per-vector scale).  Also the RMSNorm factor r (QKV,
// GU) and the per-group sums of x used to remove the +8 code offset.
// A unit (group slot gs, sequence b, k-slice j) is 16 values of x; its
// fragments fill 64 bytes: lane (c, t) of the MMA reads bytes 8 (4 c + t) of
// the slice's 64 B-byte block (c = 2b: high parts, 2b + 1: remainders), word
// 0 holding values 2t, 2t+1 and word 1 values 2t+8, 2t+9.  With INT4 weights
// every weight stage after the first of a launch finds this image already
// written by the epilogues of the stage that produced x (img_put below) and
// fetches its panel with one bulk copy; otherwise the panel's x is staged in
// the fragments' bytes and converted in place (one thread per half unit: the
// even and the odd quads of a unit read and write disjoint bytes).  This code
// runs once per stage: its loops are rolled, because each new instruction is
// fetched while the memory system carries the weight stream.  The panel's
// norm weights were copied before the stage's grid barrier (gemv_prep).
__device__ __forceinline__ uint32_t unit_offset(int gs, int b, int j, int B) {  // bytes
  return (uint32_t)gs * B * 256 + (uint32_t)(j * 2 * B + 2 * b) * 32;
}
constexpr float X_SCALE = 256.f;  // x is carried as x * 2^-8
// With an image, the norm-weight area holds the half-slice sums of the panel
// (from NW_HS_OFF, <= 8 KB) and the sums of squares of the vector (from 0,
// <= NW_HS_OFF), or the next stage's norm weights (from 0, D * 2 bytes).
constexpr int NW_HS_OFF = 24576;
static_assert(NW_HS_OFF + XF_CHUNKS * GC * 8 * 4 <= SM_NW_BYTES, "half-slice sums");

// High part and remainder of v * 2^-8 at element k of sequence b of a
// fragment image (the layout above, B sequences, slice-major): fp16 for INT4
// weights, bf16 for bf16 weights (the type of that stage's MMAs).
// Returns high part + remainder (what the MMAs multiply), for the sums below.
template <int WT>
__device__ __forceinline__ float img_put(uint8_t* img, int B, int64_t k, int b, float v) {
  const int p = (int)(k & 15), tq = (p & 7) >> 1;
  const float sv = v * (1.0f / X_SCALE);
  uint8_t* base = img + (k >> 4) * 64 * B + (p >> 3) * 4 + (p & 1) * 2 + tq * 8;
  if constexpr (WT == DDL_W_BF16) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(sv);
    const __nv_bfloat16 lo = __float2bfloat16_rn(sv - __bfloat162float(hi));
    *reinterpret_cast<__nv_bfloat16*>(base + 2 * b * 32) = hi;
    *reinterpret_cast<__nv_bfloat16*>(base + (2 * b + 1) * 32) = lo;
    return __bfloat162float(hi) + __bfloat162float(lo);
  } else {
    const __half hi = __float2half_rn(sv);
    const __half lo = __float2half_rn(sv - __half2float(hi));
    *reinterpret_cast<__half*>(base + 2 * b * 32) = hi;
    *reinterpret_cast<__half*>(base + (2 * b + 1) * 32) = lo;
    return __half2float(hi) + __half2float(lo);
  }
}
// Beside an image of K elements: per 8-element half slice and sequence, the
// sum of the fragments (high part + remainder) and the sum of squares of the
// vector itself (before the norm weight), [K / 8][B] floats each.
__device__ __forceinline__ float* img_hsum(uint8_t* img, int B, int K) {
  return reinterpret_cast<float*>(img + (((int64_t)K * 4 * B + 255) & ~int64_t(255)));
}
__device__ __forceinline__ float* img_hsq(uint8_t* img, int B, int K) { return img_hsum(img, B, K) + (K / 8) * B; }
// An epilogue's lanes (g, t), t < B, hold rows g (half slice 0) and g + 8
// (half slice 1) of a 16-row tile: the half slices' sums over g.
__device__ __forceinline__ float tile_half_sum(float v, int B) {
  const uint32_t mask = 0x11111111u * ((1u << B) - 1u);
  v += __shfl_xor_sync(mask, v, 4);
  v += __shfl_xor_sync(mask, v, 8);
  v += __shfl_xor_sync(mask, v, 16);
  return v;
}
// The image a stage writes for the next weight stage, and the one it reads.
__device__ __forceinline__ uint8_t* img_out(const Params& P, int layer, int st) {
  return P.ximg[(layer * NSTAGE + st) & 1];
}
__device__ __forceinline__ bool img_in(const Params& P, int layer, int st) {
  return P.ximg[0] != nullptr && layer * NSTAGE + st > 0;
}

template <int HD, int WT>
__device__ __forceinline__ void gemv_prologue(const Params& P, const GemvCtx& E, uint8_t* smem, Misc& M) {
  const MatGeom& m = E.m;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B;
  const int kc_lo = m.pk[E.p], nkc = m.pk[E.p + 1] - kc_lo;
  const float* x32 = nullptr;
  const uint16_t* x16 = nullptr;
  const uint16_t* nw = nullptr;  // this stage's norm weights (QKV, GU)
  const LayerDev& Ld = sp().layers[E.layer];
  switch (E.st) {
    case ST_QKV: nw = Ld.norm1; x32 = E.xin32; x16 = E.xin16; break;
    case ST_WO: x32 = P.attn; break;
    case ST_GU: x32 = P.y; nw = Ld.norm2; break;
    default: x32 = P.a; break;
  }
  const int K = m.K;
  const int ngv = (nkc - 1) * GC + chunk_groups(m, kc_lo + nkc - 1);  // group slots holding data
  const int n_units = ngv * B * 4;
  const int kbase = kc_lo * GC * DDL_GROUP;
  const bool from_img = img_in(P, E.layer, E.st);
  const uint32_t invB = (65536u + B - 1) / B;  // g / B == (g * invB) >> 16 for g < 2^15
  const uint32_t raw = smem_addr(smem + SM_SCR);
  const uint32_t nws = smem_addr(smem + SM_NW);
  // 1. copies (earlier readers of these areas, any thread, are done first):
  //    the panel of the image, or at batch 1 the panel of x as it lies in
  //    memory: one bulk copy (thread 0; the ring's copies were issued long
  //    before the barrier, so it does not queue behind them), completed on
  //    the x barrier; else quad i = (gs * B + b) * 16 + q16 of x to quad
  //    q16 % 4 of its unit.
  if (tid == 0) trace_stamp(P, E.layer * NSTAGE + E.st, NW + 4);
  csync();
  const bool bulk = from_img || (B == 1 && x32 != nullptr);
  const uint32_t xbar = smem_addr(smem + SM_XBAR), xpar = M.xuse & 1u;
  if (bulk && tid == 0) {
    fence_proxy_async_global();  // the previous stage's generic stores, read by the copy
    fence_proxy_async_smem();    // the previous stage's generic accesses to this area come first
    if (from_img) {  // the panel's fragments, its half-slice sums and (norm stages) the sums of squares
      uint8_t* src = P.ximg[(E.layer * NSTAGE + E.st - 1) & 1];
      // (bf16 weights need no sums of x: no offset to remove)
      const uint32_t ib = (uint32_t)n_units * 64, hb = WT == DDL_W_INT4 ? (uint32_t)ngv * 8 * B * 4 : 0u;
      const uint32_t qb = nw ? (uint32_t)(K / 8) * B * 4 : 0u;
      mbar_arrive_expect_tx(xbar, ib + hb + qb);
      bulk_g2s(raw, src + (int64_t)(kbase / 16) * 64 * B, ib, xbar);
      if (hb) bulk_g2s(nws + NW_HS_OFF, img_hsum(src, B, K) + (int64_t)(kbase / 8) * B, hb, xbar);
      if (qb) bulk_g2s(nws, img_hsq(src, B, K), qb, xbar);
    } else {
      mbar_arrive_expect_tx(xbar, (uint32_t)n_units * 64);
      bulk_g2s(raw, x32 + kbase, (uint32_t)n_units * 64, xbar);
    }
  }
#pragma unroll 1
  for (int i = tid; i < (bulk ? 0 : n_units * 4); i += NTHREADS) {
    const int gsb = i >> 4, q16 = i & 15;
    const int gs = (int)(((uint32_t)gsb * invB) >> 16), b = gsb - gs * B;
    const int64_t o = (int64_t)b * K + kbase + gs * DDL_GROUP + q16 * 4;
    const uint32_t dst = raw + unit_offset(gs, b, q16 >> 2, B) + (q16 & 3) * 16;
    if (x32) cp_async16(dst, x32 + o);
    else cp_async8(dst, x16 + o);
  }
  if (tid == 0) trace_stamp(P, E.layer * NSTAGE + E.st, NW + 3);
  // 2. meanwhile (norm stages without an image): the sum of squares of the
  //    whole input vector
  float* Sx = reinterpret_cast<float*>(smem + SM_SCR + XF_BYTES);
  if (nw && !from_img) {
#pragma unroll 1
    for (int b = 0; b < B; ++b) {
      float ss = 0.f;
#pragma unroll 4
      for (int q = tid; q < K / 4; q += NTHREADS) {
        const float4 x = x32 ? __ldcg(reinterpret_cast<const float4*>(x32 + (int64_t)b * K) + q)
                             : bf16x4_f32(__ldcg(reinterpret_cast<const uint2*>(x16 + (int64_t)b * K) + q));
        ss = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, ss))));
      }
      ss = warp_sum(ss);
      if (lane == 0) M.red[warp][2 * b] = ss;
    }
  }
  cp_async_wait_all();
  if (bulk && !mbar_wait_warp(xbar, xpar, P.ctrl + 1, P.wait_ns)) M.abort = 1;
  csync();
  if (bulk && tid == 0) M.xuse += 1;
  if (tid == 0) trace_stamp(P, E.layer * NSTAGE + E.st, NW + 5);
  if (from_img) {  // per (group slot, sequence) the sum of its eight half slices, in order; the sum of squares
    const float* hs = reinterpret_cast<const float*>(smem + SM_NW + NW_HS_OFF);
#pragma unroll 1
    for (int i = tid; i < (WT == DDL_W_INT4 ? ngv * B : 0); i += NTHREADS) {
      const int gs = (int)(((uint32_t)i * invB) >> 16), b = i - gs * B;
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) sum += hs[(8 * gs + q) * B + b];
      Sx[gs * NARROW_B + b] = sum;
    }
    if (nw) {
      const float* hq = reinterpret_cast<const float*>(smem + SM_NW);
#pragma unroll 1
      for (int b = 0; b < B; ++b) {
        float ss = 0.f;
        for (int q = tid; q < K / 8; q += NTHREADS) ss += hq[q * B + b];
        ss = warp_sum(ss);
        if (lane == 0) M.red[warp][2 * b] = ss;
      }
    }
  }
  // 3. conversion in place (no image): half unit h = 2 u + p of unit u holds
  //    quads p and p + 2 (values 4p..4p+3 and 4p+8..4p+11), read from bytes
  //    16p and 32 + 16p of the unit; their high parts fill bytes 16p.. and
  //    their remainders bytes 32 + 16p.., the same bytes.
  const int n_half = 2 * n_units;
  constexpr bool f16 = WT == DDL_W_INT4;
#pragma unroll 1
  for (int h = tid; h < (from_img ? 0 : n_half); h += NTHREADS) {
    const int u = h >> 1, pp = h & 1, gsb = u >> 2, j = u & 3;
    const int gs = (int)(((uint32_t)gsb * invB) >> 16);
    const uint32_t a = raw + unit_offset(gs, gsb - gs * B, j, B) + 16 * pp;
    float x[8], w[8];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float4 v;
      if (x32) {
        const uint4 r = lds128(a + 32 * q);
        v = make_float4(__uint_as_float(r.x), __uint_as_float(r.y), __uint_as_float(r.z), __uint_as_float(r.w));
      } else {
        v = bf16x4_f32(lds64(a + 32 * q));
      }
      x[4 * q] = v.x;
      x[4 * q + 1] = v.y;
      x[4 * q + 2] = v.z;
      x[4 * q + 3] = v.w;
      const uint2 wq = nw ? lds64(nws + gs * 128 + j * 32 + pp * 8 + q * 16) : make_uint2(0x3f803f80u, 0x3f803f80u);
      w[4 * q] = bf16lo_f32(wq.x);
      w[4 * q + 1] = bf16hi_f32(wq.x);
      w[4 * q + 2] = bf16lo_f32(wq.y);
      w[4 * q + 3] = bf16hi_f32(wq.y);
    }
    uint32_t hw[4], lw[4];  // word 2k + q: pair k of quad p + 2q
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int e = 4 * q + 2 * k;
        const float2 pv = make_float2(x[e] * w[e] * (1.0f / X_SCALE), x[e + 1] * w[e + 1] * (1.0f / X_SCALE));
        if (f16) {
          const __half2 hh = __float22half2_rn(pv);
          const float2 hf = __half22float2(hh);
          const __half2 ll = __float22half2_rn(make_float2(pv.x - hf.x, pv.y - hf.y));
          hw[2 * k + q] = *reinterpret_cast<const uint32_t*>(&hh);
          lw[2 * k + q] = *reinterpret_cast<const uint32_t*>(&ll);
        } else {
          const __nv_bfloat162 hh = __float22bfloat162_rn(pv);
          const float2 hf = __bfloat1622float2(hh);
          const __nv_bfloat162 ll = __float22bfloat162_rn(make_float2(pv.x - hf.x, pv.y - hf.y));
          hw[2 * k + q] = *reinterpret_cast<const uint32_t*>(&hh);
          lw[2 * k + q] = *reinterpret_cast<const uint32_t*>(&ll);
        }
      }
    sts128(a, make_uint4(hw[0], hw[1], hw[2], hw[3]));
    sts128(a + 32, make_uint4(lw[0], lw[1], lw[2], lw[3]));
  }
  if (!from_img) csync();
  // 4. (no image) per (group slot, sequence): the sum of every high part and
  //    remainder, one unit per thread, the four units of a group in adjacent
  //    lanes
#pragma unroll 1
  for (int u0 = 0; u0 < (from_img || WT != DDL_W_INT4 ? 0 : n_units); u0 += NTHREADS) {
    const int u = u0 + tid;
    float sum = 0.f;
    if (u < n_units) {
      const int gsb = u >> 2, gs = (int)(((uint32_t)gsb * invB) >> 16);
      const uint32_t a = raw + unit_offset(gs, gsb - gs * B, u & 3, B);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 r = lds128(a + 16 * q);
        const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 f;
          if (f16) f = __half22float2(*reinterpret_cast<const __half2*>(&wd[e]));
          else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[e]));
          sum += f.x + f.y;
        }
      }
    }
    sum += __shfl_xor_sync(FULL, sum, 1);
    sum += __shfl_xor_sync(FULL, sum, 2);
    if ((u & 3) == 0 && u < n_units) {
      const int gsb = u >> 2, gs = (int)(((uint32_t)gsb * invB) >> 16);
      Sx[gs * NARROW_B + (gsb - gs * B)] = sum;
    }
  }
  if (tid < B) M.escale[tid] = X_SCALE;
  // zero fragments that the stream reads for blocks past a slot's end (the
  // attention stage uses this memory too)
  for (int i = tid; i < XZ_BYTES / 4; i += NTHREADS) reinterpret_cast<uint32_t*>(smem + SM_SCR + XZ_OFF)[i] = 0u;
  if (tid == 0) trace_stamp(P, E.layer * NSTAGE + E.st, NW + 6);
  // 5. the RMSNorm factor
  csync();
  if (tid < B) {
    float ss = 0.f;
    if (nw)
      for (int w = 0; w < NW; ++w) ss += M.red[w][2 * tid];
    M.rnorm[tid] = nw ? 1.0f / sqrtf(ss / (float)K + P.eps) : 1.0f;
  }
  csync();
}

// ------------------------------------------------------------------ GEMV epilogues
// Norm weight r of the next weight stage, for the output maxima: from the copy
// that this stage's prologue staged in shared memory when the vector fits.
__device__ __forceinline__ float epi_norm(const Params& P, const uint16_t* w, int r) {
  return (int64_t)P.D * 2 <= NW_HS_OFF ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(g_smem + SM_NW)[r])
                                         : bf16_bits_to_f32(__ldg(w + r));
}

// Rows g and g+8 of tile T for sequence t (narrow batches: t = lane % 4).
template <int HD, int WT>
__device__ __noinline__ void gemv_epilogue(const Params& P, const GemvCtx& E, int T, int t, float v0,
                                           float v1, Misc& M, bool have_res = false, float res0 = 0.f,
                                           float res1 = 0.f) {
  const int lane = threadIdx.x & 31, g = lane >> 2;  // rows g, g+8 of tile T for sequence t
  if (E.st == ST_QKV) {
    const float r = M.rnorm[t];
    v0 *= r;
    v1 *= r;
    const int tph = HD / 16, head = T / tph, i = 8 * (T % tph) + g;
    if (head < P.Hq + P.Hkv) {  // RoPE on q and k: pair (i, i + hd/2)
      const float2 cs = rope_cs(P, t, i);
      const float c = cs.x, s = cs.y, a = v0, b = v1;
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
      uint16_t* row = (is_k ? E.kc : E.vc) + att_row(P, (int64_t)t * P.Hkv + kvh, seq_pos(P, t)) * HD;
      row[i] = f32_to_bf16_bits(v0);
      row[i + HD / 2] = f32_to_bf16_bits(v1);
    }
  } else if (E.st == ST_WO) {
    const int r0 = 16 * T + g, r1 = r0 + 8;
    const int64_t o = (int64_t)t * P.D;
    const float x0 = have_res ? res0 : E.xin32 ? __ldcg(E.xin32 + o + r0) : bf16_bits_to_f32(E.xin16[o + r0]);
    const float x1 = have_res ? res1 : E.xin32 ? __ldcg(E.xin32 + o + r1) : bf16_bits_to_f32(E.xin16[o + r1]);
    const float y0 = x0 + v0, y1 = x1 + v1;
    P.y[o + r0] = y0;
    P.y[o + r1] = y1;
    const uint16_t* w2 = sp().layers[E.layer].norm2;
    const float yw0 = y0 * epi_norm(P, w2, r0), yw1 = y1 * epi_norm(P, w2, r1);
    if (P.ximg[0]) {  // the gate/up stage's fragments of y * norm2, their sums, sums of y^2
      uint8_t* img = img_out(P, E.layer, E.st);
      const float p0 = img_put<WT>(img, P.B, r0, t, yw0), p1 = img_put<WT>(img, P.B, r1, t, yw1);
      const float q0 = tile_half_sum(y0 * y0, P.B), q1 = tile_half_sum(y1 * y1, P.B);
      if constexpr (WT == DDL_W_INT4) {  // the sums of x remove the INT4 code offset
        const float f0 = tile_half_sum(p0, P.B), f1 = tile_half_sum(p1, P.B);
        if (g == 0) {
          float* hs = img_hsum(img, P.B, P.D);
          hs[(2 * T) * P.B + t] = f0;
          hs[(2 * T + 1) * P.B + t] = f1;
        }
      }
      if (g == 0) {
        float* hq = img_hsq(img, P.B, P.D);
        hq[(2 * T) * P.B + t] = q0;
        hq[(2 * T + 1) * P.B + t] = q1;
      }
    } else if (P.B > NARROW_B) {  // the gate/up stage scales its staged x by this max of |y * norm2|
      atomicMax(&M.cmax[t], __float_as_uint(fmaxf(fabsf(yw0), fabsf(yw1))));
    }
  } else if (E.st == ST_GU) {
    const float r = M.rnorm[t], gt = v0 * r, up = v1 * r;
    const float av = gt / (1.0f + expf(-gt)) * up;
    P.a[(int64_t)t * P.dff + 8 * T + g] = av;
    if (P.ximg[0]) {  // the down stage's fragments of a and their sums (half slice T)
      uint8_t* img = img_out(P, E.layer, E.st);
      const float p = img_put<WT>(img, P.B, 8 * T + g, t, av);
      if constexpr (WT == DDL_W_INT4) {
        const float f = tile_half_sum(p, P.B);
        if (g == 0) img_hsum(img, P.B, P.dff)[T * P.B + t] = f;
      }
    } else if (P.B > NARROW_B) {
      atomicMax(&M.cmax[t], __float_as_uint(fabsf(av)));
    }
  } else {
    const int r0 = 16 * T + g, r1 = r0 + 8;
    const int64_t o = (int64_t)t * P.D;
    const float z0 = (have_res ? res0 : __ldcg(P.y + o + r0)) + v0, z1 = (have_res ? res1 : __ldcg(P.y + o + r1)) + v1;
    E.zout[o + r0] = z0;
    E.zout[o + r1] = z1;
    if (E.layer + 1 < P.L) {  // the next layer's QKV input: fragments of z * norm1, or their max
      const uint16_t* w1 = sp().layers[E.layer + 1].norm1;
      const float zw0 = z0 * epi_norm(P, w1, r0), zw1 = z1 * epi_norm(P, w1, r1);
      if (P.ximg[0]) {
        uint8_t* img = img_out(P, E.layer, E.st);
        const float p0 = img_put<WT>(img, P.B, r0, t, zw0), p1 = img_put<WT>(img, P.B, r1, t, zw1);
        const float q0 = tile_half_sum(z0 * z0, P.B), q1 = tile_half_sum(z1 * z1, P.B);
        if constexpr (WT == DDL_W_INT4) {
          const float f0 = tile_half_sum(p0, P.B), f1 = tile_half_sum(p1, P.B);
          if (g == 0) {
            float* hs = img_hsum(img, P.B, P.D);
            hs[(2 * T) * P.B + t] = f0;
            hs[(2 * T + 1) * P.B + t] = f1;
          }
        }
        if (g == 0) {
          float* hq = img_hsq(img, P.B, P.D);
          hq[(2 * T) * P.B + t] = q0;
          hq[(2 * T + 1) * P.B + t] = q1;
        }
      } else if (P.B > NARROW_B) {
        atomicMax(&M.cmax[t], __float_as_uint(fmaxf(fabsf(zw0), fabsf(zw1))));
      }
    }
    if (E.final_layer) {
      if (P.resid_out) {
        P.resid_out[o + r0] = z0;
        P.resid_out[o + r1] = z1;
      }
      if (P.out_bf16) {
        P.out_bf16[o + r0] = f32_to_bf16_bits(z0);
        P.out_bf16[o + r1] = f32_to_bf16_bits(z1);
      }
    }
  }
}

// Sum the partials of tile T in slot order (panel, then warp; 8 loads in
// flight) and run its epilogue.
template <int HD, int WT>
__device__ __noinline__ void gemv_fixup(const Params& P, const GemvCtx& E, int T, Misc& M) {
  const MatGeom& m = E.m;
  const int lane = threadIdx.x & 31;
  const float2* part = reinterpret_cast<const float2*>(P.gpart) + (int64_t)T * m.NP * m.J * 32 + lane;
  float s0 = 0.f, s1 = 0.f;
  for (int p = 0; p < m.NP; ++p) {  // the tile's contributors in panel p: warps v0..v1
    const uint32_t Gp = panel_groups(m, p);
    const uint32_t v0 = work_owner(m, p, (uint32_t)T * Gp, NW);
    const uint32_t v1 = work_owner(m, p, (uint32_t)(T + 1) * Gp - 1, NW);
    const float2* pp = part + (int64_t)p * m.J * 32;
#pragma unroll 4
    for (uint32_t v = v0; v <= v1; ++v) {
      if (warp_empty(m, p, v, NW)) continue;
      const float2 x = __ldcg(pp + (int64_t)(v - v0) * 32);
      s0 += x.x;
      s1 += x.y;
      *reinterpret_cast<uint64_t*>(const_cast<float2*>(pp + (int64_t)(v - v0) * 32)) = PART_EMPTY;
    }
  }
  if ((threadIdx.x & 3) < P.B) gemv_epilogue<HD, WT>(P, E, T, threadIdx.x & 3, s0, s1, M);
  if (lane == 0) P.cnt[T] = 0;
}

// Publish the partials this warp wrote: one fence, then per queued tile (on
// its own lane) add the warp's block count to the tile's counter; the warp
// that brings a counter to G finishes that tile.
template <int HD, int WT>
__device__ __noinline__ void gemv_publish(const Params& P, const GemvCtx& E, const uint32_t* pend,
                                          int npend, Misc& M) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  __threadfence();
  uint32_t last = 0;
  if (lane < npend) {
    const uint32_t T = pend[lane] & 0xFFFFFu, nblk = pend[lane] >> 20;
    last = atomicAdd(P.cnt + T, nblk) + nblk == (uint32_t)E.m.G;
  }
  uint32_t mask = __ballot_sync(FULL, last);
  if (mask) __threadfence();
  while (mask) {
    const int l = __ffs(mask) - 1;
    mask &= mask - 1;
    gemv_fixup<HD, WT>(P, E, (int)(pend[l] & 0xFFFFFu), M);
  }
}

// Cooperative launch: a tile's owner (the warp holding its first blocks in
// panel 0) finishes it.  Each other contributor stores its partial (one
// 8-byte word per lane) into a slot that holds PART_EMPTY until then, so the
// owner's polls of the slots return the partials themselves: for the warp's
// one or two owned tiles together, every lane polls its word of each
// contributor slot (bounded) until none is empty, sums the partials in slot
// order with the owner's own in its slot's place (deterministic), empties the
// slots for the next stage and runs the epilogues, whose residual inputs were
// loaded before the wait.
template <int HD, int WT>
__device__ __noinline__ void owner_fixup(const Params& P, const GemvCtx& E, int n, int T0, uint32_t mk0,
                                         float a0, float b0, int T1, uint32_t mk1, float a1, float b1,
                                         Misc& M) {
  const MatGeom& m = E.m;
  const int lane = threadIdx.x & 31, t = lane & 3, g = lane >> 2;
  if (n < 2) mk1 = 1u;  // (the owner's own slot only)
  // the residual inputs of the Wo / down epilogues
  const bool res = (E.st == ST_WO || E.st == ST_DOWN) && t < P.B && (E.st == ST_DOWN || E.xin32);
  const float* rb = E.st == ST_DOWN ? P.y : E.xin32;
  float r00 = 0.f, r01 = 0.f, r10 = 0.f, r11 = 0.f;
  if (res) {
    const int64_t o = (int64_t)t * P.D;
    r00 = __ldcg(rb + o + 16 * T0 + g);
    r01 = __ldcg(rb + o + 16 * T0 + g + 8);
    if (n > 1) {
      r10 = __ldcg(rb + o + 16 * T1 + g);
      r11 = __ldcg(rb + o + 16 * T1 + g + 8);
    }
  }
  const int64_t tstride = (int64_t)m.NP * m.J * 32;
  uint64_t* p0 = reinterpret_cast<uint64_t*>(P.gpart) + (int64_t)T0 * tstride + lane;
  uint64_t* p1 = reinterpret_cast<uint64_t*>(P.gpart) + (int64_t)(n > 1 ? T1 : T0) * tstride + lane;
  // Slots in chunks of 8 (one chunk at batch 1, more with many panels): the
  // chunk's slots are polled together and kept in registers, then summed in
  // slot order (the owner's own first) and emptied for the next stage.
  float s0 = a0, s1 = b0, u0 = a1, u1 = b1;
  const uint32_t all = mk0 | (n > 1 ? mk1 : 0u);
  uint64_t tw = 0;
#pragma unroll 1
  for (int c = 0; c < 32 && !M.abort && (all >> c) != 0u; c += 8) {
    const uint32_t own = c == 0 ? 0xFEu : 0xFFu;
    const uint32_t c0 = (mk0 >> c) & own, c1 = n > 1 ? (mk1 >> c) & own : 0u;
    uint64_t x0[8], x1[8];
#pragma unroll
    for (int f = 0; f < 8; ++f) x0[f] = x1[f] = PART_EMPTY;
    uint32_t w0 = c0, w1 = c1;
    for (uint32_t it = 1; w0 | w1; ++it) {
#pragma unroll
      for (int f = 0; f < 8; ++f) {
        if (w0 >> f & 1u) x0[f] = ld_relaxed_gpu_u64(p0 + (c + f) * 32);
        if (w1 >> f & 1u) x1[f] = ld_relaxed_gpu_u64(p1 + (c + f) * 32);
      }
#pragma unroll
      for (int f = 0; f < 8; ++f) {
        if (x0[f] != PART_EMPTY) w0 &= ~(1u << f);
        if (x1[f] != PART_EMPTY) w1 &= ~(1u << f);
      }
      if (!(w0 | w1) || (it & 63u) != 0) continue;
      const uint64_t now = globaltimer();
      if (tw == 0) tw = now;
      else if (now - tw > P.wait_ns) {
        atomicExch(P.ctrl + 1, STATUS_TIMEOUT);
        M.abort = 1;
        break;
      }
    }
#pragma unroll
    for (int f = 0; f < 8; ++f) {
      if (c0 >> f & 1u) {
        s0 += __uint_as_float((uint32_t)x0[f]);
        s1 += __uint_as_float((uint32_t)(x0[f] >> 32));
        p0[(c + f) * 32] = PART_EMPTY;
      }
      if (c1 >> f & 1u) {
        u0 += __uint_as_float((uint32_t)x1[f]);
        u1 += __uint_as_float((uint32_t)(x1[f] >> 32));
        p1[(c + f) * 32] = PART_EMPTY;
      }
    }
  }
  __syncwarp();
  if (t < P.B) {
    gemv_epilogue<HD, WT>(P, E, T0, t, s0, s1, M, res, r00, r01);
    if (n > 1) gemv_epilogue<HD, WT>(P, E, T1, t, u0, u1, M, res, r10, r11);
  }
}

// Finish this warp's share of tile T (nblk of its blocks, sums v0, v1 in true
// scale): a warp that covered the whole tile runs the epilogue directly;
// otherwise the partial goes to slot (T, panel, warp - first warp of the tile
// in the panel) and the tile is queued for publication.
template <int HD, int WT>
__device__ __forceinline__ void tile_finish(const Params& P, const GemvCtx& E, const Entry& en, Misc& M, int T,
                                            uint32_t nblk, float v0, float v1, uint32_t* pend,
                                            int& npend, int& nown, int& oT0, float& oa0, float& ob0,
                                            int& oT1, float& oa1, float& ob1) {
  const MatGeom& m = E.m;
  const int lane = threadIdx.x & 31;
  if (nblk == (uint32_t)m.G) {
    if ((threadIdx.x & 3) < P.B) gemv_epilogue<HD, WT>(P, E, T, threadIdx.x & 3, v0, v1, M);
    return;
  }
  const uint32_t me = (uint32_t)E.cl * NW + (threadIdx.x >> 5);
  const uint32_t first = T == en.T ? en.first : me;  // a later tile of the range starts in it
  if (P.cooperative && m.own_ok && E.p == 0 && me == first) {  // the tile's owner: finish it at the end
    if (nown == 0) {
      oT0 = T; oa0 = v0; ob0 = v1;
    } else if (nown == 1) {
      oT1 = T; oa1 = v0; ob1 = v1;
    } else {  // more than two (not planned for the owner path): finish this one now
      owner_fixup<HD, WT>(P, E, 1, T, owned_slots(m, T), v0, v1, 0, 0u, 0.f, 0.f, M);
      return;
    }
    ++nown;
    return;
  }
  const int64_t slot = ((int64_t)T * m.NP + E.p) * m.J + (me - first);
  if (P.cooperative && m.own_ok) {  // the tile's owner polls the slot for it
    st_relaxed_gpu_u64(reinterpret_cast<uint64_t*>(P.gpart) + slot * 32 + lane,
                       (uint64_t)__float_as_uint(v1) << 32 | __float_as_uint(v0));
    return;
  }
  reinterpret_cast<float2*>(P.gpart)[slot * 32 + lane] = make_float2(v0, v1);
  if (lane == 0) pend[npend] = (uint32_t)T | (nblk << 20);
  if (++npend == 32) {
    gemv_publish<HD, WT>(P, E, pend, npend, M);
    npend = 0;
  }
}

// Fill the CTA's stage context (thread 0); the block barrier that follows
// (the grid barrier's wait, or the one after the preparation) publishes it.
__device__ __noinline__ void fill_gemv_ctx(const Params& P, int layer, int st) {
  GemvCtx& E = ctx().E;
  if (threadIdx.x == 0) {
    E.m = sp().mg[stage_mat(st)];
    E.st = st;
    E.layer = layer;
    E.gl = P.l0 + layer;
    E.p = ctx().ent[0][st].p;
    E.cl = ctx().ent[0][st].cl;
    const LayerDev& Ld = sp().layers[layer];
    E.kc = Ld.kc;
    E.vc = Ld.vc;
    E.xin32 = nullptr;
    E.xin16 = nullptr;
    if (E.gl == 0) {
      if (P.resid_in) E.xin32 = P.resid_in;
      else E.xin16 = P.x_bf16;
    } else {
      E.xin32 = P.Z + (int64_t)((E.gl - 1) & 1) * P.B * P.D;
    }
    E.zout = P.Z + (int64_t)(E.gl & 1) * P.B * P.D;
    E.final_layer = P.final_last && layer == P.L - 1;
  }
}

// Before a weight stage's barrier: its context and the copies that do not
// depend on the previous stage (the panel's norm weights, and for Wo and down
// the next stage's norm vector for the epilogue maxima).  The copies are
// issued by warps 0..NW-2: the last warp's lane 0 made the CTA's grid-barrier
// arrival, whose release waits for the stage's writes to land.
__device__ __noinline__ void gemv_prep(const Params& P, int layer, int st, uint8_t* smem) {
  fill_gemv_ctx(P, layer, st);
  const MatGeom& m = sp().mg[stage_mat(st)];
  const int pnl = ctx().ent[0][st].p;
  const LayerDev& Ld = sp().layers[layer];
  const uint16_t* nw = st == ST_QKV ? Ld.norm1 : st == ST_GU ? Ld.norm2 : nullptr;
  const uint16_t* nw_next = st == ST_WO ? Ld.norm2
                            : (st == ST_DOWN && layer + 1 < P.L) ? sp().layers[layer + 1].norm1 : nullptr;
  if ((int64_t)P.D * 2 > NW_HS_OFF) nw_next = nullptr;
  if (img_in(P, layer, st)) nw = nullptr;  // the image carries x * norm weight already
  const int kc_lo = m.pk[pnl], nkc = m.pk[pnl + 1] - kc_lo;
  const int ngr = nkc * GC, ngv = (nkc - 1) * GC + chunk_groups(m, kc_lo + nkc - 1);
  // A whole-vector panel of QKV (after the previous layer's down stage) or of
  // gate/up (after Wo) finds its norm vector already staged, in the same
  // layout, by that weight stage's preparation for its epilogue maxima.
  if (nw && P.cooperative && nkc == m.Sk && (int64_t)P.D * 2 <= SM_NW_BYTES &&
      (st == ST_GU || layer * NSTAGE + st > P.stage_begin))
    nw = nullptr;
  const int kbase = kc_lo * GC * DDL_GROUP;
  uint8_t* nws = smem + SM_NW;
  const int nn = nw ? ngr * 8 : 0, nnx = nw_next ? P.D / 8 : 0;
  for (int i = threadIdx.x; i < nn + nnx && threadIdx.x < NTHREADS - 32; i += NTHREADS - 32) {
    if (i < nn) {
      const int gs = i >> 3, q = i & 7;
      if (gs < ngv) cp_async16(smem_addr(nws + (size_t)gs * 128 + q * 16), nw + kbase + (int64_t)gs * DDL_GROUP + q * 8);
    } else {
      const int j = i - nn;
      cp_async16(smem_addr(nws + (size_t)j * 16), nw_next + (int64_t)j * 8);
    }
  }
}

// One ring slot of a narrow-batch GEMV stage: nb blocks (groups gi.. of one
// (k-chunk, tile) unit) as PER independent MMA chains for latency hiding: the
// codes, scales and sums of x of every block first, then per k-slice j the
// blocks' x fragments and their MMAs in block order, so that consecutive MMAs
// accumulate into different blocks.  A FULL slot has PER blocks; in a partial
// one, blocks i >= nb get zero x fragments (and zero scale and sum of x), so
// they add nothing whatever stale codes the slot holds.  When another slot
// follows (`more`), its wait is made while this slot's MMAs drain.
template <int WT, int NB, bool FULL, class Wait>
__device__ __forceinline__ bool gemv_slot(const Params& P, const Ring& R, uint32_t xb, uint32_t xz, uint32_t sb,
                                          int lane, int g, int nb, bool more, float& acc0, float& acc1,
                                          Wait& wait_slot) {
  constexpr int PER = WT == DDL_W_INT4 ? BLKS_PER_SLOT : BF16_BLKS_PER_SLOT;
  constexpr uint32_t jstride = 2 * NB * 32, gstride = 4 * jstride;
  const uint32_t slot = R.slot();
  if (WT == DDL_W_INT4) {
    float c[PER][4];
    uint4 wv[PER];
    uint32_t sc[PER], xi[PER];
    float sx[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
      xi[i] = FULL || i < nb ? xb + i * gstride : xz;  // past the slot's end: zeros
      wv[i] = lds128(slot + i * QBLK_BYTES + lane * 16);
      const uint32_t scw = lds32(slot + i * QBLK_BYTES + BLK_BYTES + g * 4);
      const float sxv = lds_f32(sb + i * (NARROW_B * 4));
      sc[i] = FULL || i < nb ? scw : 0u;  // stale scale and sum words are finite-safe only as 0
      sx[i] = FULL || i < nb ? sxv : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint2 bx[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) bx[i] = lds64(xi[i] + j * jstride);
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const uint32_t w = j == 0 ? wv[i].x : j == 1 ? wv[i].y : j == 2 ? wv[i].z : wv[i].w;
        const uint32_t w8 = w >> 8;
        const uint32_t a0 = lop3_merge(w, 0x000F000Fu, 0x64086408u);
        const uint32_t a1 = lop3_merge(w, 0x00F000F0u, 0x64806480u);
        const uint32_t a2 = lop3_merge(w8, 0x000F000Fu, 0x64086408u);
        const uint32_t a3 = lop3_merge(w8, 0x00F000F0u, 0x64806480u);
        // lanes g >= 2B read unrelated fragments: they only feed C columns >= 2B, never used
        mma_f16(c[i], a0, a1, a2, a3, bx[i].x, bx[i].y);
      }
    }
    if (more && !wait_slot(R.next())) return false;
    // rows g hold 1024 + (q+8), rows g+8 hold 1024 + 16 (q+8):
    // sum q x = v - 1032 Sx  and  (v - 1152 Sx) / 16
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      acc0 = fmaf(bf16lo_f32(sc[i]), (c[i][0] + c[i][1]) - 1032.f * sx[i], acc0);
      acc1 = fmaf(bf16hi_f32(sc[i]) * 0.0625f, (c[i][2] + c[i][3]) - 1152.f * sx[i], acc1);
    }
  } else {
    float c[PER][4];
    uint2 bx[PER][4];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
      const uint32_t xi = FULL || i < nb ? xb + i * gstride : xz;  // past the slot's end: zeros
#pragma unroll
      for (int j = 0; j < 4; ++j) bx[i][j] = lds64(xi + j * jstride);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < PER; ++i) {  // stale bf16 codes could be NaN: zero them
        const uint4 av = lds128(slot + i * BF16_BLK_BYTES + j * 512 + lane * 16);
        const uint4 aq = FULL || i < nb ? av : make_uint4(0u, 0u, 0u, 0u);
        mma_bf16(c[i], aq.x, aq.y, aq.z, aq.w, bx[i][j].x, bx[i][j].y);
      }
    if (more && !wait_slot(R.next())) return false;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      acc0 += c[i][0] + c[i][1];
      acc1 += c[i][2] + c[i][3];
    }
  }
  return true;
}

// ------------------------------------------------------------------ GEMV stage
// The warp walks its range of the panel's work order (tile, k-chunk, group).
// Per ring slot (up to 8 groups of one (k-chunk, tile) unit): the 8 blocks'
// MMAs run as 8 independent chains, then fold into the unit sums; a unit's
// sums join the tile sums in true scale, and a tile is finished when the
// warp leaves it.
template <int HD, int WT, int NB>
__device__ __forceinline__ bool stage_gemv_body(const Params& P, int layer, int st, Ring& R, uint8_t* smem, Misc& M,
                                                bool wait, uint32_t target);
// The ring lives in registers while the stage runs.
template <int HD, int WT>
__device__ __noinline__ bool stage_gemv_wide(const Params& P, int layer, int st, Ring& Rm, uint8_t* smem, Misc& M);
template <int HD, int WT>
__device__ __noinline__ bool stage_gemv(const Params& P, int layer, int st, Ring& Rm, uint8_t* smem, Misc& M,
                                        bool wait, uint32_t target) {
  __syncwarp();
  Ring R = Rm;
  // the batch is a template parameter of the stream, so that the x fragments'
  // strides are constants
  const bool ok = P.B == 1   ? stage_gemv_body<HD, WT, 1>(P, layer, st, R, smem, M, wait, target)
                  : P.B == 2 ? stage_gemv_body<HD, WT, 2>(P, layer, st, R, smem, M, wait, target)
                  : P.B == 3 ? stage_gemv_body<HD, WT, 3>(P, layer, st, R, smem, M, wait, target)
                             : stage_gemv_body<HD, WT, 4>(P, layer, st, R, smem, M, wait, target);
  __syncwarp();
  Rm = R;
  __syncwarp();
  return ok;
}
template <int HD, int WT, int NB>
__device__ __forceinline__ bool stage_gemv_body(const Params& P, int layer, int st, Ring& R, uint8_t* smem, Misc& M,
                                                bool wait, uint32_t target) {
  // The grid barrier in front of the stage is waited for here, so that the
  // code after it (the prologue's copies) follows the polling loop in
  // instruction memory instead of being fetched cold once the barrier opens.
  if (wait) {
    if (!grid_wait(P, target, M)) return false;
  } else {
    csync();  // the stage context
  }
  if (threadIdx.x == 0) trace_stamp(P, layer * NSTAGE + st, 0);
  GemvCtx& E = ctx().E;  // filled by gemv_prep
  const MatGeom& m = E.m;
  gemv_prologue<HD, WT>(P, E, smem, M);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  if (threadIdx.x == 0) trace_stamp(P, layer * NSTAGE + st, 1);
  const Entry& en = ctx().ent[warp][st];
  const uint32_t lo = en.lo, hi = en.hi;
  if (lo >= hi) {
    if (lane == 0) trace_stamp(P, layer * NSTAGE + st, 2 + warp);
    return true;
  }
  uint32_t* pend = reinterpret_cast<uint32_t*>(smem + SM_SCR + XF_BYTES + SX_BYTES) + warp * 32;
  int npend = 0;
  constexpr int B = NB, B2 = 2 * B;
  const int Sk = m.Sk, pk0 = m.pk[E.p], pk1 = m.pk[E.p + 1];
  const uint32_t jstride = B2 * 32, gstride = 4 * jstride, kstride = GC * gstride;
  const uint32_t xf_lane = smem_addr(smem + SM_SCR) + (g * 4 + t) * 8;
  const uint32_t xz = smem_addr(smem + SM_SCR + XZ_OFF) + (g * 4 + t) * 8;
  const uint32_t sx_lane = smem_addr(smem + SM_SCR + XF_BYTES) + t * 4;
  const float esc = M.escale[t < B ? t : 0];
  int kc = en.kc, T = en.T, gi = en.gi, gk = en.gk;
  float acc0 = 0.f, acc1 = 0.f, tac0 = 0.f, tac1 = 0.f;
  uint32_t nblk = 0;
  int nown = 0, oT0 = 0, oT1 = 0;  // tiles this warp owns (cooperative launch), finished at the end
  float oa0 = 0.f, ob0 = 0.f, oa1 = 0.f, ob1 = 0.f;
  uint64_t wcyc = 0;  // traced: cycles waiting for the ring, slots consumed
  uint32_t nslots = 0;
  const bool tr = P.trace != nullptr;
  constexpr int PER = WT == DDL_W_INT4 ? BLKS_PER_SLOT : BF16_BLKS_PER_SLOT;
  const int glast = m.G - (Sk - 1) * m.Gc, Gc = m.Gc;  // groups of the last / other k-chunks
  // The wait for slot k + 1 is made while slot k's MMAs drain (after its
  // k-slice loop), so that a slot boundary costs no pipeline bubble.
  auto wait_slot = [&](const Ring& r) -> bool {
    const uint64_t tw = tr ? clock64() : 0;
    if (!mbar_wait_warp(r.bar(), r.phase, P.ctrl + 1, P.wait_ns)) {
      M.abort = 1;
      return false;
    }
    if (tr) wcyc += clock64() - tw;
    return true;
  };
  if (!wait_slot(R)) return false;
  // The producer cuts a unit (k-chunk kc, tile T) of the warp's range into
  // slots of PER groups from the range's first group in the unit, and a last
  // partial slot; full slots take the lean path.
  for (uint32_t b = lo; b < hi;) {
    int ng = gk - gi;  // groups of this unit in the range
    if (hi - b < (uint32_t)ng) ng = (int)(hi - b);
    const int kcl = kc - pk0;
    uint32_t xb = xf_lane + kcl * kstride + gi * gstride;
    uint32_t sb = sx_lane + ((kcl * GC + gi) * NARROW_B) * 4;
#pragma unroll 1
    for (; ng > 0;) {
      const int nb = ng < PER ? ng : PER;
      const bool more = b + nb < hi;  // another slot of this stage follows
      if (tr) ++nslots;
      const bool ok = nb == PER ? gemv_slot<WT, NB, true>(P, R, xb, xz, sb, lane, g, PER, more, acc0, acc1, wait_slot)
                                : gemv_slot<WT, NB, false>(P, R, xb, xz, sb, lane, g, nb, more, acc0, acc1, wait_slot);
      if (!ok) return false;
      ring_advance(R, lane);
      b += nb;
      gi += nb;
      nblk += nb;
      ng -= nb;
      xb += nb * gstride;
      sb += nb * (NARROW_B * 4);
    }
    if (gi == gk) {  // end of the unit: its sums join the tile's
      tac0 = fmaf(acc0, esc, tac0);
      tac1 = fmaf(acc1, esc, tac1);
      acc0 = acc1 = 0.f;
      gi = 0;
      if (++kc == pk1) {  // end of the tile in this panel
        tile_finish<HD, WT>(P, E, en, M, T, nblk, tac0, tac1, pend, npend, nown, oT0, oa0, ob0, oT1, oa1, ob1);
        tac0 = tac1 = 0.f;
        nblk = 0;
        kc = pk0;
        ++T;
      }
      gk = kc < Sk - 1 ? Gc : kc == Sk - 1 ? glast : 1;
    }
  }
  if (nblk != 0)
    tile_finish<HD, WT>(P, E, en, M, T, nblk, fmaf(acc0, esc, tac0), fmaf(acc1, esc, tac1), pend, npend, nown, oT0,
                    oa0, ob0, oT1, oa1, ob1);
  if (npend) gemv_publish<HD, WT>(P, E, pend, npend, M);
  if (nown > 0) owner_fixup<HD, WT>(P, E, nown, oT0, en.omask[0], oa0, ob0, oT1, en.omask[1], oa1, ob1, M);
  if (lane == 0) trace_stamp(P, layer * NSTAGE + st, 2 + warp);
  trace_ring(P, layer * NSTAGE + st, wcyc, nslots);
  return true;
}

// ------------------------------------------------------------------ wide batches
// Batches of NARROW_B+1..MAX_B sequences: x is carried in fp16 without the
// low part (one column per sequence, n-tile b / 8 of ntn = ceil(B / 8)), so a
// group's fragments are 4 x ntn records of 256 bytes: [j][n-tile][lane (g,t)]
// [register r] holding rows 2t, 2t+1 (r = 0) and 2t+8, 2t+9 (r = 1) of k-slice
// j for column (sequence) 8 n-tile + g.  Lane (g, t) of a tile's MMA result
// holds rows g, g+8 of sequences 8 n-tile + 2t and + 2t + 1.  The staged
// panel is at most 2 k-chunks (one for ntn = 2); per-group sums of x have a
// stride of MAX_B.  Split tiles keep 8 values per lane.
__device__ __forceinline__ int wide_ntn(int B) { return (B + 7) >> 3; }

template <int HD, int WT>
__device__ __noinline__ void gemv_prologue_wide(const Params& P, const GemvCtx& E, uint8_t* smem, Misc& M) {
  const MatGeom& m = E.m;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, ntn = wide_ntn(B);
  const int kc_lo = m.pk[E.p], nkc = m.pk[E.p + 1] - kc_lo;
  const float* x32 = nullptr;
  const uint16_t* x16 = nullptr;
  const uint16_t* nw = nullptr;
  const uint16_t* nw_next = nullptr;
  const LayerDev& Ld = sp().layers[E.layer];
  switch (E.st) {
    case ST_QKV: nw = Ld.norm1; x32 = E.xin32; x16 = E.xin16; break;
    case ST_WO: x32 = P.attn; nw_next = Ld.norm2; break;
    case ST_GU: x32 = P.y; nw = Ld.norm2; break;
    default: x32 = P.a; nw_next = E.layer + 1 < P.L ? sp().layers[E.layer + 1].norm1 : nullptr; break;
  }
  if ((int64_t)P.D * 2 > NW_HS_OFF) nw_next = nullptr;
  const int K = m.K;
  const int ngr = nkc * GC;
  const int ngv = (nkc - 1) * GC + chunk_groups(m, kc_lo + nkc - 1);
  const int kbase = kc_lo * GC * DDL_GROUP;
  const bool whole = nkc == m.Sk;
  const bool have_max = !(E.st == ST_QKV && E.layer == 0);
  uint8_t* nws = smem + SM_NW;
  csync();
  float xm = 0.f;
  if (have_max && tid < B) xm = __uint_as_float(__ldcg(P.xmax + (E.layer * NSTAGE + E.st) * MAX_B + tid));
  if (nw && !whole) {
    for (int b = 0; b < B; ++b) {
      float ss = 0.f;
      for (int q = tid; q < K / 4; q += NTHREADS) {
        const float4 v = x32 ? __ldcg(reinterpret_cast<const float4*>(x32 + (int64_t)b * K) + q)
                             : bf16x4_f32(__ldcg(reinterpret_cast<const uint2*>(x16 + (int64_t)b * K) + q));
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
      }
      ss = warp_sum(ss);
      if (lane == 0) M.red[warp][2 * b] = ss;
    }
  }
  cp_async_wait_all();
  csync();
  // item it = ((group slot * B + b) * 16 + quad): four columns of sequence b, read from memory
#define WIDE_X(it_, gs_, b_, q16_)                                                                         \
  (x32 ? __ldcg(reinterpret_cast<const float4*>(x32 + (int64_t)(b_) * K + kbase + (gs_) * DDL_GROUP) + (q16_)) \
       : bf16x4_f32(__ldcg(reinterpret_cast<const uint2*>(x16 + (int64_t)(b_) * K + kbase + (gs_) * DDL_GROUP) + (q16_))))
  if (!have_max) {  // first layer of a launch: the panel's max per sequence
    for (int b = 0; b < B; ++b) {
      float mx = 0.f;
      for (int it = tid; it < ngr * 16; it += NTHREADS) {
        const int gs = it >> 4, q16 = it & 15;
        if (gs >= ngv) continue;
        float4 x = WIDE_X(it, gs, b, q16);
        if (nw) {
          const float4 w = bf16x4_f32(*reinterpret_cast<const uint2*>(nws + (size_t)gs * 128 + q16 * 8));
          x = make_float4(x.x * w.x, x.y * w.y, x.z * w.z, x.w * w.w);
        }
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
      }
      mx = warp_max(mx);
      if (lane == 0) M.red[warp][2 * b + 1] = mx;
    }
    csync();
    if (tid < B)
      for (int w = 0; w < NW; ++w) xm = fmaxf(xm, M.red[w][2 * tid + 1]);
  }
  if (tid < B) {
    const int e = xm > 0.f ? ilogbf(xm) - 11 : 0;
    M.escale[tid] = ldexpf(1.0f, e);
    M.edown[tid] = ldexpf(1.0f, -e);
  }
  csync();
  // fragments (fp16 of x * w * 2^-e) and the sum of x per (group, sequence);
  // the sum of squares per sequence when the panel is the whole vector
  uint32_t* xf = reinterpret_cast<uint32_t*>(smem + SM_SCR);
  float* Sx = reinterpret_cast<float*>(smem + SM_SCR + XF_BYTES);
  constexpr bool f16 = WT == DDL_W_INT4;
  const bool want_ss = nw && whole;
  const int gwords = 4 * ntn * 64;  // 32-bit words of one group's fragments
  // sequence by sequence (item = group slot * 16 + quad), so that the sums
  // of squares reduce in a fixed order
  for (int b = 0; b < B; ++b) {
    const float sc = M.edown[b];
    float ssb = 0.f;
    for (int base = warp * 32; base < ngr * 16; base += 4 * NTHREADS) {
      float4 x[4];
      bool ok[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = base + u * NTHREADS + lane, gs = it >> 4, q16 = it & 15;
        ok[u] = it < ngr * 16 && gs < ngv;
        x[u] = ok[u] ? WIDE_X(it, gs, b, q16) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = base + u * NTHREADS + lane, gs = it >> 4, q16 = it & 15;
        float part = 0.f;
        if (ok[u]) {
          if (want_ss) ssb = fmaf(x[u].x, x[u].x, fmaf(x[u].y, x[u].y, fmaf(x[u].z, x[u].z, fmaf(x[u].w, x[u].w, ssb))));
          const float4 w = nw ? bf16x4_f32(*reinterpret_cast<const uint2*>(nws + (size_t)gs * 128 + q16 * 8))
                              : make_float4(1.f, 1.f, 1.f, 1.f);
          const float v0 = x[u].x * w.x * sc, v1 = x[u].y * w.y * sc, v2 = x[u].z * w.z * sc, v3 = x[u].w * w.w * sc;
          uint32_t h01, h23;
          float2 f01, f23;
          if (f16) {
            const __half2 a = __float22half2_rn(make_float2(v0, v1)), c = __float22half2_rn(make_float2(v2, v3));
            f01 = __half22float2(a);
            f23 = __half22float2(c);
            h01 = *reinterpret_cast<const uint32_t*>(&a);
            h23 = *reinterpret_cast<const uint32_t*>(&c);
          } else {
            const __nv_bfloat162 a = __float22bfloat162_rn(make_float2(v0, v1));
            const __nv_bfloat162 c = __float22bfloat162_rn(make_float2(v2, v3));
            f01 = __bfloat1622float2(a);
            f23 = __bfloat1622float2(c);
            h01 = *reinterpret_cast<const uint32_t*>(&a);
            h23 = *reinterpret_cast<const uint32_t*>(&c);
          }
          part = (f01.x + f01.y) + (f23.x + f23.y);
          const int j = q16 >> 2, reg = (q16 >> 1) & 1, t0 = 2 * (q16 & 1), nt = b >> 3, g = b & 7;
          uint32_t* f = xf + gs * gwords + (j * ntn + nt) * 64;
          f[(g * 4 + t0) * 2 + reg] = h01;
          f[(g * 4 + t0 + 1) * 2 + reg] = h23;
        }
#pragma unroll
        for (int o = 8; o; o >>= 1) part += __shfl_xor_sync(FULL, part, o);
        if (q16 == 0 && ok[u]) Sx[gs * MAX_B + b] = part;
      }
    }
    if (want_ss) {
      ssb = warp_sum(ssb);
      if (lane == 0) M.red[warp][2 * b] = ssb;
    }
  }
#undef WIDE_X
  for (int i = tid; i < XZ_BYTES / 4; i += NTHREADS) reinterpret_cast<uint32_t*>(smem + SM_SCR + XZ_OFF)[i] = 0u;
  csync();
  if (tid < B) {
    float ss = 0.f;
    if (nw)
      for (int w = 0; w < NW; ++w) ss += M.red[w][2 * tid];
    M.rnorm[tid] = nw ? 1.0f / sqrtf(ss / (float)K + P.eps) : 1.0f;
  }
  csync();
}

// Split tiles of a wide batch: 8 values per lane, float4 x 2 at [slot][lane].
template <int HD>
__device__ __forceinline__ void wide_epilogues(const Params& P, const GemvCtx& E, int T, const float (&v)[8],
                                               Misc& M) {
  const int t = threadIdx.x & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int b = nt * 8 + 2 * t + s;
      if (b < P.B) gemv_epilogue<HD, DDL_W_INT4>(P, E, T, b, v[nt * 4 + s], v[nt * 4 + 2 + s], M);  // (INT4 only)
    }
}
template <int HD>
__device__ __forceinline__ void wide_sum_slots(const Params& P, const GemvCtx& E, int T, float (&v)[8]) {
  const MatGeom& m = E.m;
  const int lane = threadIdx.x & 31;
  const float4* part = reinterpret_cast<const float4*>(P.gpart) + (int64_t)T * m.NP * m.J * 64 + lane * 2;
#pragma unroll
  for (int k = 0; k < 8; ++k) v[k] = 0.f;
  for (int p = 0; p < m.NP; ++p) {
    const uint32_t Gp = panel_groups(m, p);
    const uint32_t v0 = work_owner(m, p, (uint32_t)T * Gp, NW), v1 = work_owner(m, p, (uint32_t)(T + 1) * Gp - 1, NW);
    for (uint32_t w = v0; w <= v1; ++w) {
      if (warp_empty(m, p, w, NW)) continue;
      const float4* q = part + ((int64_t)p * m.J + (w - v0)) * 64;
      const float4 a = __ldcg(q), c = __ldcg(q + 1);
      v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
      v[4] += c.x; v[5] += c.y; v[6] += c.z; v[7] += c.w;
    }
  }
}
// Cooperative launch: the owner waits for the other contributors' releases,
// then sums the partial slots in `mask` (its own included) in slot order.
template <int HD>
__device__ __noinline__ void wide_owner_fixup(const Params& P, const GemvCtx& E, int T, uint32_t mask, Misc& M) {
  const MatGeom& m = E.m;
  const int lane = threadIdx.x & 31;
  const uint32_t expected = __popc(mask) - 1;
  if (lane == 0) {
    uint64_t t0 = 0;
    for (uint32_t it = 1; ld_acquire_gpu(P.cnt + T) < expected; ++it) {
      if ((it & 255u) != 0) continue;
      const uint64_t now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > P.wait_ns) {
        atomicExch(P.ctrl + 1, STATUS_TIMEOUT);
        M.abort = 1;
        break;
      }
    }
  }
  __syncwarp();
  float v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) v[k] = 0.f;
  const float4* part = reinterpret_cast<const float4*>(P.gpart) + (int64_t)T * m.NP * m.J * 64 + lane * 2;
  for (uint32_t r = mask; r; r &= r - 1) {
    const float4* q = part + (int64_t)(__ffs(r) - 1) * 64;
    const float4 a = __ldcg(q), c = __ldcg(q + 1);
    v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
    v[4] += c.x; v[5] += c.y; v[6] += c.z; v[7] += c.w;
  }
  wide_epilogues<HD>(P, E, T, v, M);
  if (lane == 0) P.cnt[T] = 0;
}
// One launch per stage: the warp whose arrival completes the tile finishes it.
template <int HD>
__device__ __noinline__ void wide_publish(const Params& P, const GemvCtx& E, const uint32_t* pend, int npend,
                                          Misc& M) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  __threadfence();
  uint32_t last = 0;
  if (lane < npend) {
    const uint32_t T = pend[lane] & 0xFFFFFu, nblk = pend[lane] >> 20;
    last = atomicAdd(P.cnt + T, nblk) + nblk == (uint32_t)E.m.G;
  }
  uint32_t mask = __ballot_sync(FULL, last);
  if (mask) __threadfence();
  while (mask) {
    const int l = __ffs(mask) - 1;
    mask &= mask - 1;
    const int T = (int)(pend[l] & 0xFFFFFu);
    float v[8];
    wide_sum_slots<HD>(P, E, T, v);
    wide_epilogues<HD>(P, E, T, v, M);
    if (lane == 0) P.cnt[T] = 0;
  }
}
template <int HD>
__device__ __forceinline__ void wide_tile_finish(const Params& P, const GemvCtx& E, const Entry& en, Misc& M, int T,
                                                 uint32_t nblk,
                                                 const float (&v)[8], uint32_t* pend, int& npend, int& nown,
                                                 int& oT0, int& oT1) {
  const MatGeom& m = E.m;
  const int lane = threadIdx.x & 31;
  if (nblk == (uint32_t)m.G) {
    wide_epilogues<HD>(P, E, T, v, M);
    return;
  }
  const uint32_t me = (uint32_t)E.cl * NW + (threadIdx.x >> 5);
  const uint32_t first = T == en.T ? en.first : me;  // a later tile of the range starts in it
  const int64_t slot = ((int64_t)T * m.NP + E.p) * m.J + (me - first);
  float4* q = reinterpret_cast<float4*>(P.gpart) + slot * 64 + lane * 2;
  q[0] = make_float4(v[0], v[1], v[2], v[3]);
  q[1] = make_float4(v[4], v[5], v[6], v[7]);
  if (P.cooperative && m.own_ok) {
    if (E.p == 0 && me == first) {  // the owner: finish at the end (its own partial is in its slot)
      if (nown == 0) oT0 = T;
      else if (nown == 1) oT1 = T;
      if (nown >= 2) {  // more than two (not planned for the owner path): finish this one now
        __syncwarp();
        wide_owner_fixup<HD>(P, E, T, owned_slots(m, T), M);
        return;
      }
      ++nown;
      return;
    }
    __syncwarp();
    if (lane == 0) red_release_gpu_add(P.cnt + T, 1u);
    return;
  }
  if (lane == 0) pend[npend] = (uint32_t)T | (nblk << 20);
  if (++npend == 32) {
    wide_publish<HD>(P, E, pend, npend, M);
    npend = 0;
  }
}

template <int HD, int WT>
__device__ __noinline__ bool stage_gemv_wide(const Params& P, int layer, int st, Ring& Rm, uint8_t* smem, Misc& M) {
  __syncwarp();
  Ring R = Rm;
  GemvCtx& E = ctx().E;  // filled by gemv_prep
  const MatGeom& m = E.m;
  gemv_prologue_wide<HD, WT>(P, E, smem, M);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  if (threadIdx.x == 0) trace_stamp(P, layer * NSTAGE + st, 1);
  const Entry& en = ctx().ent[warp][st];
  const uint32_t lo = en.lo, hi = en.hi;
  bool ok = true;
  if (lo < hi) {
    uint32_t* pend = reinterpret_cast<uint32_t*>(smem + SM_SCR + XF_BYTES + SX_BYTES) + warp * 32;
    int npend = 0;
    const int B = P.B, ntn = wide_ntn(B), Sk = m.Sk, pk0 = m.pk[E.p], pk1 = m.pk[E.p + 1];
    const uint32_t jstride = ntn * 256, gstride = 4 * jstride, kstride = GC * gstride;
    const uint32_t xf_lane = smem_addr(smem + SM_SCR) + (g * 4 + t) * 8;
    const uint32_t xz = smem_addr(smem + SM_SCR + XZ_OFF) + (g * 4 + t) * 8;
    const uint32_t sx0 = smem_addr(smem + SM_SCR + XF_BYTES);
    float esc[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int b = nt * 8 + 2 * t + s;
        esc[nt][s] = b < B ? M.escale[b] : 0.f;
      }
    int kc = en.kc, T = en.T, gi = en.gi, gk = en.gk;
    float acc[8], tac[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = tac[k] = 0.f;
    uint32_t nblk = 0;
    int nown = 0, oT0 = 0, oT1 = 0;
    constexpr int PER = WT == DDL_W_INT4 ? BLKS_PER_SLOT : BF16_BLKS_PER_SLOT;
    constexpr int HB = PER >= 4 ? 2 : 1;
    for (uint32_t b = lo; b < hi;) {
      int nb = (int)(hi - b < (uint32_t)PER ? hi - b : (uint32_t)PER);
      if (nb > gk - gi) nb = gk - gi;
      const uint32_t slot = R.slot();
      if (!mbar_wait_warp(R.bar(), R.phase, P.ctrl + 1, P.wait_ns)) {
        M.abort = 1;
        ok = false;
        break;
      }
      const int kcl = kc - pk0;
      const uint32_t xb = xf_lane + kcl * kstride + gi * gstride;
      const int gsl = kcl * GC + gi;  // group slot of the slot's first block
#pragma unroll 1
      for (int h0 = 0; h0 < PER; h0 += HB) {
        float c[HB][2][4];
        uint2 bx[HB][4][2];
#pragma unroll
        for (int ii = 0; ii < HB; ++ii) {
          const int i = h0 + ii;
          const uint32_t xi = i < nb ? xb + i * gstride : xz;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            c[ii][nt][0] = c[ii][nt][1] = c[ii][nt][2] = c[ii][nt][3] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              bx[ii][j][nt] = nt < ntn ? lds64(xi + (j * ntn + nt) * 256) : make_uint2(0u, 0u);
          }
        }
        if (WT == DDL_W_INT4) {
          uint4 wv[HB];
          uint32_t sc[HB];
          float sx[HB][2][2];
#pragma unroll
          for (int ii = 0; ii < HB; ++ii) {
            const int i = h0 + ii;
            wv[ii] = lds128(slot + i * QBLK_BYTES + lane * 16);
            const uint32_t scw = lds32(slot + i * QBLK_BYTES + BLK_BYTES + g * 4);
            sc[ii] = i < nb ? scw : 0u;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int s = 0; s < 2; ++s) {
                const int bq = nt * 8 + 2 * t + s;
                const float v = lds_f32(sx0 + ((gsl + (i < nb ? i : 0)) * MAX_B + bq) * 4);
                sx[ii][nt][s] = (i < nb && bq < B) ? v : 0.f;
              }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int ii = 0; ii < HB; ++ii) {
              const uint32_t w = j == 0 ? wv[ii].x : j == 1 ? wv[ii].y : j == 2 ? wv[ii].z : wv[ii].w;
              const uint32_t w8 = w >> 8;
              const uint32_t a0 = lop3_merge(w, 0x000F000Fu, 0x64086408u);
              const uint32_t a1 = lop3_merge(w, 0x00F000F0u, 0x64806480u);
              const uint32_t a2 = lop3_merge(w8, 0x000F000Fu, 0x64086408u);
              const uint32_t a3 = lop3_merge(w8, 0x00F000F0u, 0x64806480u);
              mma_f16(c[ii][0], a0, a1, a2, a3, bx[ii][j][0].x, bx[ii][j][0].y);
              if (ntn > 1) mma_f16(c[ii][1], a0, a1, a2, a3, bx[ii][j][1].x, bx[ii][j][1].y);
            }
          }
#pragma unroll
          for (int ii = 0; ii < HB; ++ii) {
            const float slo = bf16lo_f32(sc[ii]), shi = bf16hi_f32(sc[ii]) * 0.0625f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int s = 0; s < 2; ++s) {
                acc[nt * 4 + s] = fmaf(slo, c[ii][nt][s] - 1032.f * sx[ii][nt][s], acc[nt * 4 + s]);
                acc[nt * 4 + 2 + s] = fmaf(shi, c[ii][nt][2 + s] - 1152.f * sx[ii][nt][s], acc[nt * 4 + 2 + s]);
              }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int ii = 0; ii < HB; ++ii) {
              const int i = h0 + ii;
              const uint4 av = lds128(slot + i * BF16_BLK_BYTES + j * 512 + lane * 16);
              const uint4 aq = i < nb ? av : make_uint4(0u, 0u, 0u, 0u);
              mma_bf16(c[ii][0], aq.x, aq.y, aq.z, aq.w, bx[ii][j][0].x, bx[ii][j][0].y);
              if (ntn > 1) mma_bf16(c[ii][1], aq.x, aq.y, aq.z, aq.w, bx[ii][j][1].x, bx[ii][j][1].y);
            }
#pragma unroll
          for (int ii = 0; ii < HB; ++ii)
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] += c[ii][k >> 2][k & 3];
        }
      }
      ring_advance(R, lane);
      b += nb;
      gi += nb;
      nblk += nb;
      if (gi == gk) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          tac[k] = fmaf(acc[k], esc[k >> 2][k & 1], tac[k]);
          acc[k] = 0.f;
        }
        gi = 0;
        if (++kc == pk1) {
          wide_tile_finish<HD>(P, E, en, M, T, nblk, tac, pend, npend, nown, oT0, oT1);
#pragma unroll
          for (int k = 0; k < 8; ++k) tac[k] = 0.f;
          nblk = 0;
          kc = pk0;
          ++T;
        }
        gk = kc < Sk ? chunk_groups(m, kc) : 1;
      }
    }
    if (ok) {
      if (nblk != 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) tac[k] = fmaf(acc[k], esc[k >> 2][k & 1], tac[k]);
        wide_tile_finish<HD>(P, E, en, M, T, nblk, tac, pend, npend, nown, oT0, oT1);
      }
      if (npend) wide_publish<HD>(P, E, pend, npend, M);
      __syncwarp();
      if (nown > 0) wide_owner_fixup<HD>(P, E, oT0, en.omask[0], M);
      if (nown > 1) wide_owner_fixup<HD>(P, E, oT1, en.omask[1], M);
    }
  }
  if (lane == 0) trace_stamp(P, layer * NSTAGE + st, 2 + warp);
  __syncwarp();
  Rm = R;
  __syncwarp();
  return ok;
}

// ------------------------------------------------------------------ attention
// Merge head h of the CTA's shared softmax records (m, l, o; fp32 records of
// GH*(hd+2) padded to REC floats) into `out`: record `first`, then record 2v
// of every warp v in vmask.  M = max m_k, f_k = exp2(m_k - M),
// l = sum f_k l_k, o = sum f_k o_k.  Lane d handles head dims d, d+32, ...
template <int HD>
__device__ __forceinline__ void merge_head(const float* recs, int REC, int first, uint32_t vmask,
                                           float* out, int GH, int h) {
  const int lane = threadIdx.x & 31;
  float mx = recs[first * REC + GH * HD + h];
  for (uint32_t mm = vmask; mm; mm &= mm - 1)
    mx = fmaxf(mx, recs[2 * (__ffs(mm) - 1) * REC + GH * HD + h]);
  const float mref = mx == -INFINITY ? 0.f : mx;  // records without keys (m = -inf) weigh 0
  float acc[HD / 32], l = 0.f;
#pragma unroll
  for (int dd = 0; dd < HD / 32; ++dd) acc[dd] = 0.f;
  int ri = first;
  for (uint32_t mm = vmask;;) {
    const float* r = recs + ri * REC;
    const float f = exp2f(r[GH * HD + h] - mref);
    l = fmaf(f, r[GH * HD + GH + h], l);
#pragma unroll
    for (int dd = 0; dd < HD / 32; ++dd) acc[dd] = fmaf(f, r[h * HD + lane + 32 * dd], acc[dd]);
    if (!mm) break;
    ri = 2 * (__ffs(mm) - 1);
    mm &= mm - 1;
  }
#pragma unroll
  for (int dd = 0; dd < HD / 32; ++dd) out[h * HD + lane + 32 * dd] = acc[dd];
  if (lane == 0) {
    out[GH * HD + h] = mx;
    out[GH * HD + GH + h] = l;
  }
}

// Final merge of all CTA records of one sequence into attn, by the last CTA
// to finish it; it is on the stage's critical path, so its loads go out in
// one round trip.  Thread (h, d-quad) first copies (cp.async) its o column of
// the first 2 NW records into the CTA's record area of shared memory, free by
// now; meanwhile (phase 1) warp h < GH folds every record's (m, l) of head h
// into per-record factors exp2(m_j - M) / L (one round trip for up to 64
// records).  Phase 2: the thread sums factor * o over the records (any past
// 2 NW from global memory in rounds of 8).  A record whose factor is 0 (a
// CTA without tiles holds none) is skipped, whatever its memory holds.
template <int HD, int WT>
__device__ __noinline__ void merge_sequence(const Params& P, int layer, int64_t seq, int64_t Ta, int64_t C,
                                            int64_t cf, int n, float* stage, float* fac, Misc& M) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int GH = P.GH, REC = att_rec_floats(GH, HD);
  const float* base = P.apart + seq * P.J_att * REC;
  // with more tiles than CTAs every CTA of the sequence holds a record; with
  // fewer, a CTA whose tile range is empty holds none
  const bool all_full = Ta >= C;
  constexpr int DQ = HD / 4;  // float4 columns of a head; GH * DQ <= NTHREADS (MAX_GH = 8)
  constexpr int MV = 2 * NW;  // records staged in shared memory (their o parts fill <= 2 NW REC floats)
  const int e = threadIdx.x, h = e / DQ, dq = e - h * DQ;
  const bool act = h < GH;
  const int nst = n < MV ? n : MV;
  if (act)
    for (int u = 0; u < nst; ++u)
      cp_async16(smem_addr(stage + (u * GH + h) * HD + 4 * dq), base + (int64_t)u * REC + h * HD + 4 * dq);
  if (warp < GH) {
    // one round trip for the (m, l) of up to 64 records per lane pair
    float mj[2], lj[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int j = lane + 32 * u;
      const bool ok = j < n && (all_full || range_lo(Ta, C, cf + j) != range_lo(Ta, C, cf + j + 1));
      mj[u] = ok ? __ldcg(base + (int64_t)j * REC + GH * HD + warp) : -INFINITY;
      lj[u] = ok ? __ldcg(base + (int64_t)j * REC + GH * HD + GH + warp) : 0.f;
    }
    for (int j0 = 64; j0 < n; j0 += 32) {  // more than 64 CTAs per sequence: the rest
      const int j = j0 + lane;
      const bool ok = j < n && (all_full || range_lo(Ta, C, cf + j) != range_lo(Ta, C, cf + j + 1));
      if (ok) mj[0] = fmaxf(mj[0], __ldcg(base + (int64_t)j * REC + GH * HD + warp));
    }
    const float mx = warp_max(fmaxf(mj[0], mj[1]));
    float l = 0.f;
    for (int j = lane; j < n; j += 32) {
      float fj = 0.f;
      if (j < 64) {
        const float m = j < 32 ? mj[0] : mj[1];
        fj = m == -INFINITY ? 0.f : exp2f(m - mx);
        l = fmaf(fj, j < 32 ? lj[0] : lj[1], l);
      } else if (all_full || range_lo(Ta, C, cf + j) != range_lo(Ta, C, cf + j + 1)) {
        const float* rec = base + (int64_t)j * REC;
        fj = exp2f(__ldcg(rec + GH * HD + warp) - mx);
        l = fmaf(fj, __ldcg(rec + GH * HD + GH + warp), l);
      }
      fac[warp * P.J_att + j] = fj;
    }
    l = warp_sum(l);
    for (int j = lane; j < n; j += 32) fac[warp * P.J_att + j] /= l;
  }
  cp_async_wait_all();
  csync();
  const int64_t b = seq / P.Hkv, kvh = seq % P.Hkv;
  float fsum = 0.f;
  if (act) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](float fj, float4 x) {
      if (fj != 0.f) {
        acc.x = fmaf(fj, x.x, acc.x);
        acc.y = fmaf(fj, x.y, acc.y);
        acc.z = fmaf(fj, x.z, acc.z);
        acc.w = fmaf(fj, x.w, acc.w);
      }
    };
#pragma unroll 4
    for (int u = 0; u < nst; ++u)
      add(fac[h * P.J_att + u], *reinterpret_cast<const float4*>(stage + (u * GH + h) * HD + 4 * dq));
#pragma unroll 1
    for (int j0 = MV; j0 < n; j0 += 8) {
      float4 w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        w[u] = j0 + u < n ? __ldcg(reinterpret_cast<const float4*>(base + (int64_t)(j0 + u) * REC + h * HD) + dq)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 8; ++u) add(j0 + u < n ? fac[h * P.J_att + j0 + u] : 0.f, w[u]);
    }
    float* dst = P.attn + b * P.Hq * HD + (kvh * GH + h) * HD;
    reinterpret_cast<float4*>(dst)[dq] = acc;
    if (P.ximg[0]) {  // the Wo stage's fragments of the attention output
      uint8_t* img = img_out(P, layer, ST_ATT);
      const int64_t k = (kvh * GH + h) * HD + 4 * dq;
      float f = img_put<WT>(img, P.B, k, (int)b, acc.x);
      f += img_put<WT>(img, P.B, k + 1, (int)b, acc.y);
      f += img_put<WT>(img, P.B, k + 2, (int)b, acc.z);
      f += img_put<WT>(img, P.B, k + 3, (int)b, acc.w);
      fsum = f;
    } else if (P.B > NARROW_B) {  // the Wo stage scales its staged x by this
      const float m = fmaxf(fmaxf(fabsf(acc.x), fabsf(acc.y)), fmaxf(fabsf(acc.z), fabsf(acc.w)));
      if (b < MAX_B) atomicMax(&M.cmax[b], __float_as_uint(m));
    }
  }
  // the half slice's other four elements are thread dq ^ 1's (the next lane);
  // (bf16 weights need no sums of x)
  if constexpr (WT == DDL_W_INT4) {
    fsum += __shfl_xor_sync(FULL, fsum, 1);
    if (P.ximg[0] && act && (dq & 1) == 0) {
      const int64_t k = (kvh * GH + h) * HD + 4 * dq;
      img_hsum(img_out(P, layer, ST_ATT), P.B, P.Hq * HD)[(k >> 3) * P.B + b] = fsum;
    }
  }
  csync();
}

// Write one warp's softmax state (m, l, o) for its current sequence segment:
// to the CTA's record slot 0 (first segment) or 1 (last), or, for a segment
// wholly inside the warp, straight to the sequence's partial of this CTA.
template <int HD>
__device__ __forceinline__ void att_flush(const Params& P, float* rec, const float (&o)[HD / 8][4],
                                          float mrun, float lrun) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3, GH = P.GH;
  float ls = lrun + __shfl_xor_sync(FULL, lrun, 1);
  ls += __shfl_xor_sync(FULL, ls, 2);
  if (g < GH) {
#pragma unroll
    for (int nb = 0; nb < HD / 8; ++nb) {
      rec[g * HD + 8 * nb + 2 * t] = o[nb][0] + o[nb][2];
      rec[g * HD + 8 * nb + 2 * t + 1] = o[nb][1] + o[nb][3];
    }
    if (t == 0) {
      rec[GH * HD + g] = mrun;
      rec[GH * HD + GH + g] = ls;
    }
  }
}

template <int HD, int WT, bool RAG>
__device__ __forceinline__ bool stage_att_body(const Params& P, int layer, Ring& R, uint8_t* smem, Misc& M);
// The stage waits for its grid barrier itself (wait) or for the CTA's other
// warps, so that its own code is being fetched while the barrier completes.
template <int HD, int WT, bool RAG>
__device__ __noinline__ bool stage_att(const Params& P, int layer, Ring& Rm, uint8_t* smem, Misc& M, bool wait,
                                       uint32_t target) {
  if (wait) {
    if (!grid_wait(P, target, M)) return false;
  } else {
    csync();  // the stage context
  }
  if (threadIdx.x == 0) {
    trace_stamp(P, layer * NSTAGE + ST_ATT, 0);
    trace_stamp(P, layer * NSTAGE + ST_ATT, 1);
  }
  __syncwarp();
  Ring R = Rm;
  const bool ok = stage_att_body<HD, WT, RAG>(P, layer, R, smem, M);
  __syncwarp();
  Rm = R;
  __syncwarp();
  return ok;
}
template <int HD, int WT, bool RAG>
__device__ __forceinline__ bool stage_att_body(const Params& P, int layer, Ring& R, uint8_t* smem, Misc& M) {
  constexpr int KS = HD / 16, NB = HD / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int GH = P.GH, REC = att_rec_floats(GH, HD), nt = P.nt_att;
  const int64_t Ta = (int64_t)P.B * P.Hkv * nt, C = gridDim.x;
  const LayerDev& Ld = sp().layers[layer];
  const AttCta& A = ctx().att;
  float* recs = reinterpret_cast<float*>(smem + SM_SCR);
  const int64_t lo = ctx().ent[warp][ST_ATT].lo, hi = ctx().ent[warp][ST_ATT].hi;
  const float qscale = 1.4426950408889634f / sqrtf((float)HD);  // log2(e) / sqrt(hd)
  int nseg = 0;
  int64_t first_seq = -1, cur = -1;
  uint32_t qa[KS][4];
  float mrun = -INFINITY, lrun = 0.f;
  float o[NB][4];
  bool ok = true, kready = false;
  uint64_t wcyc = 0;  // traced: cycles waiting for the ring, slots consumed
  uint32_t nslots = 0;
  int64_t pq = P.pos;  // the current sequence's position and its tiles holding keys
  int ntq = nt;

  for (int64_t it = lo; it < hi && ok; ++it) {
    const int64_t seq = (uint32_t)it / (uint32_t)nt;
    const int i = (int)((uint32_t)it - (uint32_t)seq * (uint32_t)nt);
    if (seq != cur) {
      if (cur >= 0)  // a segment wholly inside this warp (or the warp's first)
        att_flush<HD>(P, nseg == 1 ? recs + (warp * 2) * REC
                                   : P.apart + (cur * P.J_att + (blockIdx.x - A.cf[cur - A.s0])) * REC,
                      o, mrun, lrun);
      cur = seq;
      ++nseg;
      if constexpr (RAG) {  // this sequence's position and tiles holding keys
        pq = P.posb[seq / P.Hkv];
        ntq = (int)(pq / 16) + 1;
      }
      if (first_seq < 0) first_seq = seq;
      const int b = (int)(seq / P.Hkv), kvh = (int)(seq % P.Hkv);
      const float* qp = P.q + (int64_t)b * P.Hq * HD + (int64_t)(kvh * GH + g) * HD;
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        float2 v0 = make_float2(0.f, 0.f), v1 = make_float2(0.f, 0.f);
        if (g < GH) {
          v0 = __ldcg(reinterpret_cast<const float2*>(qp + 16 * j + 2 * t));
          v1 = __ldcg(reinterpret_cast<const float2*>(qp + 16 * j + 2 * t + 8));
        }
        const float v[4] = {v0.x * qscale, v0.y * qscale, v1.x * qscale, v1.y * qscale};
        float h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          h[e] = __bfloat162float(__float2bfloat16_rn(v[e]));
          l[e] = v[e] - h[e];
        }
        qa[j][0] = pack_bf16x2(h[0], h[1]);  // rows g: high part
        qa[j][1] = pack_bf16x2(l[0], l[1]);  // rows g+8: low part
        qa[j][2] = pack_bf16x2(h[2], h[3]);
        qa[j][3] = pack_bf16x2(l[2], l[3]);
      }
      mrun = -INFINITY;
      lrun = 0.f;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
    }
    if (i >= ntq) {  // past the sequence's new token (its record stays empty): the next sequence
      it = (seq + 1) * nt - 1;
      continue;
    }
    // K of this tile in slot R, V in the slot after it.  The K slot goes back
    // to the producer once the scores are computed, and the wait for the
    // next tile's K is made while the P.V MMAs drain.
    const uint32_t ks = R.slot();
    if (!kready) {
      const uint64_t tw = P.trace ? clock64() : 0;
      if (!mbar_wait_warp(R.bar(), R.phase, P.ctrl + 1, P.wait_ns)) {
        M.abort = 1;
        ok = false;
        break;
      }
      if (P.trace) wcyc += clock64() - tw;
    }
    if (P.trace) nslots += 2;
    const bool newtok = i == ntq - 1;  // the tile holding the new token
    const int rnew = (int)(pq - 16 * (int64_t)i);
    // Rows of the tile written by this step's QKV stage, possibly after the
    // producer's copy: the new token's, and in a prefill every prompt row from
    // p0 on (the rows share one cache).  They are reloaded from the cache, and
    // the rows after the new token zeroed; these generic writes come before
    // the slot's next bulk (async-proxy) fill.
    int r_lo = rnew, r_hi = rnew;
    int64_t ro = ((seq * P.s_max) + pq) * HD;  // the new token's row in the cache ([seq][s_max][hd])
    bool fix = newtok;
    if constexpr (RAG) {
      ro = att_row(P, seq, 16 * (int64_t)i) * HD;  // the tile's first row
      r_hi = newtok ? rnew : 15;
      if (P.p0 >= 0) {
        const int64_t lo = P.p0 - 16 * (int64_t)i;
        r_lo = lo > 0 ? (int)lo : 0;
        fix = 16 * (int64_t)i + 15 >= P.p0;
      }
    }
    auto patch = [&](uint32_t sl, const uint16_t* cache) {
      if constexpr (RAG) {
        const int n = (r_hi - r_lo + 1) * (HD / 8);
        for (int z = lane; z < n; z += 32) {
          const int r = r_lo + z / (HD / 8), ch = z % (HD / 8);
          sts128(kv_addr(sl, r, ch), ldcg_u128(cache + ro + (int64_t)r * HD + ch * 8));
        }
      } else {
        if (lane < HD / 8) sts128(kv_addr(sl, rnew, lane), ldcg_u128(cache + ro + lane * 8));
      }
      if (newtok) {
        const int nz = (15 - rnew) * (HD / 8);
        for (int z = lane; z < nz; z += 32)
          sts128(kv_addr(sl, rnew + 1 + z / (HD / 8), z % (HD / 8)), make_uint4(0u, 0u, 0u, 0u));
      }
      fence_proxy_async_smem();
      __syncwarp();
    };
    if (fix) patch(ks, Ld.kc);
    // scores: rows g = high-part dot products, rows g+8 = low-part ones
    float s[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int jj = 0; jj < KS; jj += 2) {
        const int mat = lane >> 3, r = lane & 7;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kv_addr(ks, 8 * n + r, 2 * (jj + (mat >> 1)) + (mat & 1)), b0, b1, b2, b3);
        mma_bf16(s[n], qa[jj][0], qa[jj][1], qa[jj][2], qa[jj][3], b0, b1);
        mma_bf16(s[n], qa[jj + 1][0], qa[jj + 1][1], qa[jj + 1][2], qa[jj + 1][3], b2, b3);
      }
    }
    ring_advance(R, lane);  // the K slot: its rows are in registers now
    const uint32_t vs = R.slot();
    {
      const uint64_t tw = P.trace ? clock64() : 0;
      if (!mbar_wait_warp(R.bar(), R.phase, P.ctrl + 1, P.wait_ns)) {
        M.abort = 1;
        ok = false;
        break;
      }
      if (P.trace) wcyc += clock64() - tw;
    }
    if (fix) patch(vs, Ld.vc);
    // online softmax over this tile (score of key 8n + 2t + e = s[n][e] + s[n][e+2])
    float sv[2][2];
    float mt = -INFINITY;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int64_t key = 16 * (int64_t)i + 8 * n + 2 * t + e;
        sv[n][e] = key > pq ? -INFINITY : s[n][e] + s[n][e + 2];
        mt = fmaxf(mt, sv[n][e]);
      }
    mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 2));
    const float mnew = fmaxf(mrun, mt);
    const float alpha = exp2f(mrun - mnew);
    float ph[2][2], pl[2][2], psum = 0.f;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float p = exp2f(sv[n][e] - mnew);
        psum += p;
        ph[n][e] = __bfloat162float(__float2bfloat16_rn(p));
        pl[n][e] = p - ph[n][e];
      }
    lrun = lrun * alpha + psum;
    mrun = mnew;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      o[nb][0] *= alpha;
      o[nb][1] *= alpha;
      o[nb][2] *= alpha;
      o[nb][3] *= alpha;
    }
    const uint32_t pa0 = pack_bf16x2(ph[0][0], ph[0][1]), pa1 = pack_bf16x2(pl[0][0], pl[0][1]);
    const uint32_t pa2 = pack_bf16x2(ph[1][0], ph[1][1]), pa3 = pack_bf16x2(pl[1][0], pl[1][1]);
    // o rows g += p_hi V, rows g+8 += p_lo V  (head dims 8nb + 2t, +1)
#pragma unroll
    for (int nb = 0; nb < NB; nb += 2) {
      const int mat = lane >> 3, r = lane & 7;
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(kv_addr(vs, 8 * (mat & 1) + r, nb + (mat >> 1)), b0, b1, b2, b3);
      mma_bf16(o[nb], pa0, pa1, pa2, pa3, b0, b1);
      mma_bf16(o[nb + 1], pa0, pa1, pa2, pa3, b2, b3);
    }
    kready = false;
    int64_t nx = it + 1;  // the next tile holding keys: the next one, or the next sequence's first
    if (RAG && nx < hi && nx - seq * nt >= ntq) nx = (seq + 1) * nt;
    if (nx < hi) {  // the next tile's K, while these MMAs drain
      const Ring Rk = R.next();
      const uint64_t tw = P.trace ? clock64() : 0;
      if (!mbar_wait_warp(Rk.bar(), Rk.phase, P.ctrl + 1, P.wait_ns)) {
        M.abort = 1;
        ok = false;
        break;
      }
      if (P.trace) wcyc += clock64() - tw;
      kready = true;
    }
    ring_advance(R, lane);  // the V slot
  }
  if (ok && nseg > 0) att_flush<HD>(P, recs + (warp * 2 + (nseg == 1 ? 0 : 1)) * REC, o, mrun, lrun);
  if (lane == 0) trace_stamp(P, layer * NSTAGE + ST_ATT, 2 + warp);
  trace_ring(P, layer * NSTAGE + ST_ATT, wcyc, nslots);
  if (lane == 0) {
    M.seg_n[warp] = ok ? nseg : 0;
    M.seg_first[warp] = first_seq;
    M.seg_last[warp] = cur;
  }
  csync();
  if (M.abort) return false;
  // CTA merge: runs of consecutive warp records of one sequence (found by
  // thread 0), each merged head by head with the heads spread over the warps
  if (threadIdx.x == 0) {
    int nr = 0;
    for (int w = 0; w < NW; ++w) {
      const int n = M.seg_n[w];
      if (n == 0) continue;
      if (nr > 0 && M.run_seq[nr - 1] == M.seg_first[w]) {
        M.run_vmask[nr - 1] |= 1u << w;  // record 2w continues the open run
      } else {
        M.run_seq[nr] = M.seg_first[w];
        M.run_first[nr] = 2 * w;
        M.run_vmask[nr] = 0u;
        ++nr;
      }
      if (n > 1) {  // the warp's last segment starts a new run (record 2w+1)
        M.run_seq[nr] = M.seg_last[w];
        M.run_first[nr] = 2 * w + 1;
        M.run_vmask[nr] = 0u;
        ++nr;
      }
    }
    for (int r = 0; r < nr; ++r)
      M.run_out[r] = (M.run_seq[r] * P.J_att + (blockIdx.x - A.cf[M.run_seq[r] - A.s0])) * REC;
    M.nruns = nr;
  }
  csync();
  for (int r = 0; r < M.nruns; ++r)
    for (int h = warp; h < GH; h += NW)
      merge_head<HD>(recs, REC, M.run_first[r], M.run_vmask[r], P.apart + M.run_out[r], GH, h);
  // the last CTA to publish a sequence's record merges the sequence
  csync();
  if (A.ns > 0) {
    const int64_t s0 = A.s0, s1 = A.s0 + A.ns - 1;
    if (threadIdx.x <= s1 - s0) {  // one thread per sequence: the arrivals in flight together
      const int64_t sq = s0 + threadIdx.x;
      const uint32_t n = A.n[threadIdx.x];
      const uint32_t old = atom_add_acq_rel(P.seqcnt + sq, 1u);
      M.mseq[threadIdx.x] = old == n - 1 ? sq : -1;
      if (old == n - 1) P.seqcnt[sq] = 0;
    }
    csync();
    float* fac = recs + NW * 2 * REC;  // per (head, record) factors of the merge
    for (int64_t sq = s0; sq <= s1; ++sq)
      if (M.mseq[(int)(sq - s0)] == sq)
        merge_sequence<HD, WT>(P, layer, sq, Ta, C, A.cf[sq - s0], A.span[sq - s0], recs, fac, M);
  }
  return true;
}

// This CTA's maximum of its stage output (times the consumer's norm weight)
// to the consumer stage's word, for sequence threadIdx.x.
__device__ __noinline__ void flush_cmax(const Params& P, Misc& M, int layer, int st) {
  const int cl = st == ST_DOWN ? layer + 1 : layer;
  const int cs = st == ST_ATT ? ST_WO : st == ST_WO ? ST_GU : st == ST_GU ? ST_DOWN : ST_QKV;
  if (st != ST_QKV && cl < P.L && M.cmax[threadIdx.x] != 0u)
    atomicMax(P.xmax + (cl * NSTAGE + cs) * MAX_B + threadIdx.x, M.cmax[threadIdx.x]);
  M.cmax[threadIdx.x] = 0u;
}

// ------------------------------------------------------------------ producer
// Lane w (< NW) of the producer warp fills consumer warp w's ring: it walks
// the warp's slots of every stage of the launch with its own cursor and
// issues slot n as soon as the consumer handed slot n - DEPTH back.  It polls
// without blocking (the lanes' rings advance independently) and naps between
// rounds that find nothing to do, stops when the consumers abort or when no
// ring advanced for the wait limit, and before leaving waits for its copies
// in flight, so that none lands after the CTA has gone.
template <int HD, int WT, bool RAG>
__device__ __noinline__ void producer(const Params& P, uint8_t* smem, Misc& M) {
  const int lane = threadIdx.x & 31;
  const uint64_t policy = policy_evict_first();
  const uint32_t slot0 = smem_addr(smem + SM_RING + lane * DEPTH * SLOT_BYTES);
  const uint32_t fbar0 = smem_addr(smem + SM_BARS + lane * DEPTH * 8);
  const uint32_t ebar0 = smem_addr(smem + SM_EBARS + lane * DEPTH * 8);
  Cursor c;
  SlotDesc d;
  bool have = false;
  if (lane < NW) {
    c.s = P.stage_begin;
    cursor_enter<WT, RAG>(P, c, lane);
    have = cursor_next<WT, RAG>(P, c, lane, d);
  }
  uint32_t n = 0;  // slots issued
  uint64_t t0 = 0;
  bool stop = false;
#pragma unroll 1
  for (uint32_t it = 1; __any_sync(FULL, have); ++it) {
    bool moved = false;
    if (have && (n < DEPTH || mbar_test_wait(ebar0 + (n % DEPTH) * 8, ((n / DEPTH) + 1) & 1))) {
      issue_slot<HD, WT>(c, d, slot0 + (n % DEPTH) * SLOT_BYTES, fbar0 + (n % DEPTH) * 8, policy);
      ++n;
      have = cursor_next<WT, RAG>(P, c, lane, d);
      moved = true;
    }
    if (__any_sync(FULL, moved)) {
      t0 = 0;
      continue;
    }
    // Nothing to issue: a short pause, so that the polling takes few issue
    // slots from the consumer warps that share this warp's scheduler.
    __nanosleep(PRODUCER_NAP_NS);
    if ((it & 15u) != 0) continue;
    if (*reinterpret_cast<volatile int*>(&M.abort)) stop = true;
    const uint64_t now = globaltimer();
    if (t0 == 0) t0 = now;
    else if (now - t0 > P.wait_ns) {
      if (lane == 0) atomicExch(P.ctrl + 1, STATUS_TIMEOUT);
      stop = true;
    }
    if (__any_sync(FULL, stop)) break;
  }
  // copies in flight: the last DEPTH slots issued on each ring (bounded)
  if (lane < NW) {
    const uint64_t t1 = globaltimer();
    for (uint32_t k = n > DEPTH ? n - DEPTH : 0; k < n; ++k)
      while (!mbar_test_wait(fbar0 + (k % DEPTH) * 8, (k / DEPTH) & 1))
        if (globaltimer() - t1 > P.wait_ns) break;
  }
}

// ------------------------------------------------------------------ the kernel
template <int HD, int WT, bool WIDE, bool RAG>
__global__ void __launch_bounds__(NTHREADS_ALL, 1) decode_kernel(const __grid_constant__ Params P) {
  uint8_t* smem = g_smem;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  {  // indexed parameters to shared memory (read after the barrier below)
    SParams& S = *reinterpret_cast<SParams*>(smem + SM_SPAR);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(P.mg);
    uint32_t* dst = reinterpret_cast<uint32_t*>(S.mg);
    for (int i = threadIdx.x; i < (int)(sizeof(S.mg) / 4); i += NTHREADS_ALL) dst[i] = src[i];
    src = reinterpret_cast<const uint32_t*>(P.rope);
    dst = reinterpret_cast<uint32_t*>(S.rope);
    for (int i = threadIdx.x; i < (int)(sizeof(S.rope) / 4); i += NTHREADS_ALL) dst[i] = src[i];
    src = reinterpret_cast<const uint32_t*>(P.layers);
    dst = reinterpret_cast<uint32_t*>(S.layers);
    const int nw32 = P.L * (int)(sizeof(LayerDev) / 4);
    for (int i = threadIdx.x; i < nw32; i += NTHREADS_ALL) dst[i] = src[i];
  }
  Misc& M = *reinterpret_cast<Misc*>(smem + SM_MISC);
  if (warp < NW) {
    Ring& R = ctx().ring[warp];  // warp-uniform: every lane writes the same values
    R.slot0 = smem_addr(smem + SM_RING + warp * DEPTH * SLOT_BYTES);
    R.bar0 = smem_addr(smem + SM_BARS + warp * DEPTH * 8);
    R.ebar0 = smem_addr(smem + SM_EBARS + warp * DEPTH * 8);
    R.idx = 0;
    R.phase = 0;
    if (lane < DEPTH) {
      mbar_init(R.bar0 + lane * 8, 1);
      mbar_init(R.ebar0 + lane * 8, 1);
    }
  }
  if (threadIdx.x == 0) {
    M.abort = 0;
    M.xuse = 0;
    mbar_init(smem_addr(smem + SM_XBAR), 1);
  }
  if (threadIdx.x < MAX_B) M.cmax[threadIdx.x] = 0u;
  mbar_init_fence();
  __syncthreads();
  // Roles.  A non-inlined function must not be called on both sides of the
  // register split, so the consumers compute the work entries after theirs
  // and publish them to the producer through barrier 2.
  if (warp >= NW) {  // the producer warpgroup
    regs_dec<PRODUCER_REGS>();
    if (warp == NW) {
      asm volatile("bar.sync 2, %0;" ::"n"(NTHREADS + 32) : "memory");
      producer<HD, WT, RAG>(P, smem, M);
    }
    return;
  }
  regs_inc<CONSUMER_REGS>();
  compute_entries(P);
  asm volatile("bar.arrive 2, %0;" ::"n"(NTHREADS + 32) : "memory");
  csync();  // every warp's entries written before any warp reads another's (the stage context reads warp 0's)
  // A launch that overlaps the previous kernel (the tensor-core path's
  // attention stage) waits for it here; the producer does not: it reads only
  // weights and K/V history, and the consumers reload the rows this step
  // appends.
  pdl_wait();
  Ring& R = ctx().ring[warp];
  bool ok = true;
  for (int s = P.stage_begin; s < P.stage_end && ok; ++s) {
    const int layer = s / NSTAGE, st = s % NSTAGE;
    if (st != ST_ATT) gemv_prep(P, layer, st, smem);
    // (a held barrier waits for one arrival more than the grid makes: its
    // bounded wait gives up and the call reports a timeout)
    const bool wait = s != P.stage_begin && P.cooperative;
    const uint32_t target = (uint32_t)(s - P.stage_begin) * gridDim.x + (P.l0 * NSTAGE + s == P.hold_stage);
    if (st != ST_ATT && !WIDE) {  // the narrow GEMV stage waits for its barrier itself
      stage_gemv<HD, WT>(P, layer, st, R, smem, M, wait, target);
      if (M.abort) {
        ok = false;
        break;
      }
    } else if (st == ST_ATT) {
      ok = stage_att<HD, WT, RAG>(P, layer, R, smem, M, wait, target);
      if (!ok) break;
    } else {
      if (wait) {
        if (!grid_wait(P, target, M)) {
          ok = false;
          break;
        }
      } else {
        csync();  // the stage context
      }
      if (threadIdx.x == 0) trace_stamp(P, s, 0);
      stage_gemv_wide<HD, WT>(P, layer, st, R, smem, M);
    }
    csync();
    if (threadIdx.x == 0) trace_stamp(P, s, NW + 2);
    if (M.abort) ok = false;
    if (threadIdx.x < P.B && threadIdx.x < MAX_B) flush_cmax(P, M, layer, st);
    if (P.cooperative && s + 1 < P.stage_end) grid_arrive(P);
  }
  if (!ok) {
    cp_async_wait_all();  // this thread's copies in flight (the stage preparation's) land first
    if (threadIdx.x == 0) M.abort = 1;  // the producer stops and waits for its copies
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
static uint64_t g_wait_ns = WAIT_LIMIT_NS;  // limit of every bounded device wait
static int g_hold_stage = -1;  // test hook: the grid barrier before this flattened stage never completes
static uint64_t* g_trace = nullptr;
static size_t g_trace_bytes = 0;

template <int HD, int WT>
static int prepare_kernel() {
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (done[dev]) return DDL_OK;
  if constexpr (WT == DDL_W_INT4) {  // the wide-batch variant
    for (const void* f : {(const void*)decode_kernel<HD, WT, true, false>, (const void*)decode_kernel<HD, WT, true, true>}) {
      cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SM_TOTAL);
      if (e != cudaSuccess) return cuda_status(e);
    }
  }
  for (const void* f : {(const void*)decode_kernel<HD, WT, false, false>, (const void*)decode_kernel<HD, WT, false, true>}) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SM_TOTAL);
    if (e != cudaSuccess) return cuda_status(e);
  }
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
  int64_t ctrl, cnt, seqcnt, xmax, gpart, apart, Z, q, attn, y, a, rope, ptab, ximg, ximg_bytes, tc, total;
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
    const int64_t u = (int64_t)mg[k].NT * mg[k].NP * mg[k].J * 32 * (B > NARROW_B ? 8 : 2) * 4;
    if (u > gpart) gpart = u;
    if (mg[k].NT > ntmax) ntmax = mg[k].NT;
  }
  int64_t off = 0;
  w.ctrl = off;  off = align256(off + 256);
  w.cnt = off;   off = align256(off + ntmax * 4);
  w.seqcnt = off; off = align256(off + (int64_t)B * s.H_kv * 4);
  w.xmax = off;  off = align256(off + (int64_t)MAX_LAYERS * NSTAGE * MAX_B * 4);
  w.gpart = off; off = align256(off + gpart);
  w.apart = off; off = align256(off + (int64_t)B * s.H_kv * (Jatt + 1) * att_rec_floats(GH, s.head_dim) * 4);
  w.Z = off;     off = align256(off + 2 * (int64_t)B * s.D * 4);
  w.q = off;     off = align256(off + (int64_t)B * Nq * 4);
  w.attn = off;  off = align256(off + (int64_t)B * Nq * 4);
  w.y = off;     off = align256(off + (int64_t)B * s.D * 4);
  w.a = off;     off = align256(off + (int64_t)B * s.d_ff * 4);
  w.rope = off;  off = align256(off + (int64_t)B * (64 * 2 * 4 + 4));  // ragged positions: RoPE table, positions
  w.ptab = off;  off = align256(off + (int64_t)B * ((s_max + 15) / 16) * 4);  // page table (pages >= 16 slots)
  // fragment images of a weight stage's input (fp16 high part and remainder
  // per element), two by stage parity; batches up to IMG_MAX_B
  int64_t kmax = s.D > s.d_ff ? s.D : s.d_ff;
  if (Nq > kmax) kmax = Nq;
  w.ximg = off;
  w.ximg_bytes = B <= IMG_MAX_B ? align256(kmax * 4 * B) + align256(2 * (kmax / 8) * B * 4) : 0;
  off += 2 * w.ximg_bytes;
  w.tc = off;  // the tensor-core path's partials, operand images and sums (batches past NARROW_B)
  if (B > NARROW_B) off = align256(off + tc_workspace_bytes(s, B, DDL_W_INT4));
  w.total = off;
}

static int plan(const ddl_shape* s, int wtype, int B, int64_t s_max, int C, MatGeom mg[4],
                WsLayout& w) {
  make_geoms(*s, wtype, mg);
  for (int k = 0; k < 4; ++k) {
    if (mg[k].T * (int64_t)C >= (int64_t(1) << 32) || mg[k].NT >= (1 << 20))
      return DDL_ERR_UNSUPPORTED;  // 32-bit work-split arithmetic, 20-bit tile ids
    if (!make_panels(mg[k], B, C)) return DDL_ERR_UNSUPPORTED;
  }
  ws_layout(*s, B, s_max, C, mg, w);
  return DDL_OK;
}

// cuTensorMapEncodeTiled from the driver, found once through the runtime.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  });
  return fn;
}
// The [rows][hd] bf16 view of a K or V cache for 16-row x 64-column boxes
// with the 128-byte swizzle (rows = B * H_kv * s_max).
static int encode_kv_map(CUtensorMap* m, const uint16_t* base, int64_t rows, int hd) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return DDL_ERR_CUDA;
  const cuuint64_t dims[2] = {(cuuint64_t)hd, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)hd * 2};
  const cuuint32_t box[2] = {64, 16};  // 16 rows x 128 bytes: one half of an hd-128 row (all of hd 64)
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dims, strides,
                         box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DDL_OK : DDL_ERR_CUDA;
}

// RoPE table of sequences at their own positions (fp64 angles, as the host
// computes the shared one), and the positions as int32 for the epilogues.
struct RopeFill {
  int32_t posb[64];
  double base;
  int32_t hd, B;
  float* table;   // [B][64][2]
  int32_t* pos;   // [B]
};
__global__ void rope_fill_kernel(const __grid_constant__ RopeFill R) {
  const int b = blockIdx.x, i = threadIdx.x;
  if (b >= R.B) return;
  if (i < R.hd / 2) {
    const double phi = (double)R.posb[b] * pow(R.base, -2.0 * i / (double)R.hd);
    R.table[((int64_t)b * 64 + i) * 2] = (float)cos(phi);
    R.table[((int64_t)b * 64 + i) * 2 + 1] = (float)sin(phi);
  }
  if (i == 0) R.pos[b] = R.posb[b];
}

// A paged cache: host page table [rows][per_seq], the page size (a power of
// two >= 16) and the pool's page count.
struct Paged {
  const int32_t* table;
  int32_t per_seq, page_size;
  int64_t pages;
};

// Page-table checks: every live entry (the pages of slots 0 .. pos of each
// table row in use) names a page of the pool, and every page that receives a
// new row occurs once among them: no other sequence reads it and its own
// sequence does not map it twice.  Prefill (shared) uses row 0 for all rows.
static int check_pages(const Paged& pg, int32_t B, const int64_t* posv, bool shared) {
  const int rows = shared ? 1 : B;
  std::unordered_map<int32_t, int> seen;
  for (int r = 0; r < rows; ++r) {
    const int64_t last = shared ? posv[B - 1] : posv[r];
    for (int64_t j = 0; j <= last / pg.page_size; ++j) {
      const int32_t id = pg.table[(int64_t)r * pg.per_seq + j];
      if (id < 0 || id >= pg.pages) return DDL_ERR_ARG;
      ++seen[id];
    }
  }
  for (int r = 0; r < rows; ++r) {
    const int64_t first = shared ? posv[0] : posv[r], last = shared ? posv[B - 1] : posv[r];
    for (int64_t j = first / pg.page_size; j <= last / pg.page_size; ++j)
      if (seen[pg.table[(int64_t)r * pg.per_seq + j]] != 1) return DDL_ERR_ARG;
  }
  return DDL_OK;
}

// posv: NULL (every sequence at pos) or a host array of B positions (pos unused).
// shared: the B rows are one sequence's consecutive tokens on one cache (prefill).
// pg: paged caches (with posv), else NULL.
static int decode(const ddl_shape* s, ddl_wtype wtype, const ddl_layer_w* layers, const ddl_kv* kv,
                  int32_t L, int32_t B, int64_t pos, const float* resid_in, const uint16_t* x_bf16,
                  float* resid_out, uint16_t* out_bf16, void* workspace, size_t ws_bytes,
                  void* stream, const int64_t* posv = nullptr, bool shared = false, const Paged* pg = nullptr) {
  int st = check_shape(s);
  if (st) return st;
  if (!layers || !kv || L <= 0 || !workspace) return !workspace ? DDL_ERR_WORKSPACE : DDL_ERR_ARG;
  if (B < 1 || B > TC_MAX_B) return DDL_ERR_UNSUPPORTED;
  if (wtype != DDL_W_INT4 && wtype != DDL_W_BF16) return DDL_ERR_UNSUPPORTED;
  // the weight stages on the tcgen05 tensor cores: INT4 from TC_MIN_B
  // sequences on, bf16 past NARROW_B (whose warp-level MMAs would need bf16
  // activations, 8 bits, which miss the tolerance)
  const bool use_tc = (wtype == DDL_W_INT4 && B >= TC_MIN_B) || (wtype == DDL_W_BF16 && B > NARROW_B);
  if (!resid_in && !x_bf16) return DDL_ERR_ARG;
  const int64_t s_max = kv[0].s_max;
  // rows of a layer's cache view (the TMA tensor map's outer dimension, 32-bit in the kernel)
  const int64_t kv_rows = pg ? pg->pages * s->H_kv * pg->page_size : (shared ? 1 : (int64_t)B) * s->H_kv * s_max;
  if (kv_rows >= (1ll << 31) || (int64_t)B * s->H_kv * s_max >= (1ll << 31)) return DDL_ERR_UNSUPPORTED;
  if (posv) {  // the largest position sets the attention's tile count
    pos = 0;
    for (int b = 0; b < B; ++b) {
      if (posv[b] < 0 || posv[b] >= s_max) return DDL_ERR_POS;
      if (posv[b] > pos) pos = posv[b];
    }
  }
  if (pos < 0 || pos >= s_max) return DDL_ERR_POS;
  if (pg && (!posv || (st = check_pages(*pg, B, posv, shared)))) return posv ? st : DDL_ERR_ARG;
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
  if ((st = plan(s, wtype, B, s_max, C, P.mg, w))) return st;
  if ((int64_t)ws_bytes < w.total) return DDL_ERR_WORKSPACE;
  const int HD = s->head_dim;
  st = HD == 128 ? (wtype == DDL_W_INT4 ? prepare_kernel<128, DDL_W_INT4>() : prepare_kernel<128, DDL_W_BF16>())
                 : (wtype == DDL_W_INT4 ? prepare_kernel<64, DDL_W_INT4>() : prepare_kernel<64, DDL_W_BF16>());
  if (st) return st;
  if (use_tc && wtype == DDL_W_BF16)  // its attention stage runs on the INT4 wide-batch instance
    if ((st = HD == 128 ? prepare_kernel<128, DDL_W_INT4>() : prepare_kernel<64, DDL_W_INT4>())) return st;
  uint8_t* ws = (uint8_t*)workspace;
  P.D = s->D; P.Hq = s->H_q; P.Hkv = s->H_kv; P.hd = HD; P.dff = s->d_ff; P.B = B;
  P.GH = s->H_q / s->H_kv; P.eps = s->eps; P.wtype = wtype; P.rope_base = s->rope_base;
  P.pos = pos; P.s_max = s_max;
  P.kv_bstride = shared ? 0 : (int64_t)s->H_kv * s_max;
  P.p0 = -1;
  P.wait_ns = g_wait_ns;
  P.hold_stage = g_hold_stage;
  P.nt_att = (int32_t)((pos + 1 + 15) / 16);
  for (int i = 0; i < HD / 2; ++i) {  // RoPE angles in fp64: pos * base^(-2i/hd)
    const double phi = (double)pos * pow(s->rope_base, -2.0 * i / (double)HD);
    P.rope[i][0] = (float)cos(phi);
    P.rope[i][1] = (float)sin(phi);
  }
  P.J_att = (int32_t)att_J((int64_t)B * s->H_kv, P.nt_att, C);
  // shared scratch of the attention merges: 2 records per warp + the factors
  if ((int64_t)(NW * 2 * att_rec_floats(P.GH, HD) + P.GH * P.J_att) * 4 > SM_SCR_BYTES) return DDL_ERR_UNSUPPORTED;
  {  // a CTA's attention range may touch at most 8 sequences
    const int64_t Ta = (int64_t)B * s->H_kv * P.nt_att, per = (Ta + C - 1) / C;
    if ((per + P.nt_att - 1) / P.nt_att + 1 > 8) return DDL_ERR_UNSUPPORTED;
  }
  P.resid_in = resid_in; P.x_bf16 = x_bf16; P.resid_out = resid_out; P.out_bf16 = out_bf16;
  P.ctrl = (uint32_t*)(ws + w.ctrl); P.cnt = (uint32_t*)(ws + w.cnt);
  P.seqcnt = (uint32_t*)(ws + w.seqcnt);
  P.xmax = (uint32_t*)(ws + w.xmax);
  P.gpart = (float*)(ws + w.gpart); P.apart = (float*)(ws + w.apart); P.Z = (float*)(ws + w.Z);
  P.q = (float*)(ws + w.q); P.attn = (float*)(ws + w.attn); P.y = (float*)(ws + w.y);
  P.a = (float*)(ws + w.a);
  P.ximg[0] = P.ximg[1] = nullptr;
  if (w.ximg_bytes > 0 && (int64_t)s->D / 8 * B * 4 <= NW_HS_OFF) {  // (batches up to IMG_MAX_B)
    P.ximg[0] = ws + w.ximg;
    P.ximg[1] = ws + w.ximg + w.ximg_bytes;
  }
  cudaStream_t cs = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(ws, 0, (size_t)w.gpart, cs);  // barrier, status, counters
  if (e != cudaSuccess) return cuda_status(e);
  if (posv) {
    RopeFill rf;
    memset(&rf, 0, sizeof rf);
    for (int b = 0; b < B; ++b) rf.posb[b] = (int32_t)posv[b];
    rf.base = s->rope_base;
    rf.hd = HD;
    rf.B = B;
    rf.table = (float*)(ws + w.rope);
    rf.pos = (int32_t*)(ws + w.rope + (int64_t)B * 64 * 2 * 4);
    rope_fill_kernel<<<B, 64, 0, cs>>>(rf);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);
    P.ragged = 1;
    for (int b = 0; b < B; ++b) P.posb[b] = (int32_t)posv[b];
    P.p0 = shared ? (int32_t)posv[0] : -1;
    P.rope_b = rf.table;
  }
  if (pg) {  // the page table rows in use, to the workspace (the host copy may go once this returns)
    const size_t n = (size_t)(shared ? 1 : B) * pg->per_seq * 4;
    if ((e = cudaMemcpyAsync(ws + w.ptab, pg->table, n, cudaMemcpyHostToDevice, cs)) != cudaSuccess)
      return cuda_status(e);
    P.ptab = (const int32_t*)(ws + w.ptab);
    P.pshift = 0;
    while ((1 << P.pshift) < pg->page_size) ++P.pshift;
    P.pstride = shared ? 0 : pg->per_seq;
  }
  // empty partial slots (each reader empties the slots it consumed, so they
  // stay empty from stage to stage within a launch)
  if ((e = cudaMemsetAsync(ws + w.gpart, 0xFF, (size_t)(w.apart - w.gpart), cs)) != cudaSuccess)
    return cuda_status(e);
  const bool coop = di.coop && g_launch_mode == 0 && !use_tc;
  const bool wide = B > NARROW_B;  // INT4, or only the attention stage (tensor-core path)
  // (bf16 weights past NARROW_B run only the attention stage, on the INT4 wide instance)
  const int wsel = (wide || wtype == DDL_W_INT4) ? DDL_W_INT4 : DDL_W_BF16;
  void* fn = nullptr;
#define DDL_PICK(HDV, WTV, WIDEV)                                                                           \
  fn = posv ? (void*)decode_kernel<HDV, WTV, WIDEV, true> : (void*)decode_kernel<HDV, WTV, WIDEV, false>
  if (HD == 128) {
    if (wide) DDL_PICK(128, DDL_W_INT4, true);
    else if (wsel == DDL_W_INT4) DDL_PICK(128, DDL_W_INT4, false);
    else DDL_PICK(128, DDL_W_BF16, false);
  } else {
    if (wide) DDL_PICK(64, DDL_W_INT4, true);
    else if (wsel == DDL_W_INT4) DDL_PICK(64, DDL_W_INT4, false);
    else DDL_PICK(64, DDL_W_BF16, false);
  }
#undef DDL_PICK
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
      if ((st = encode_kv_map(&P.kmap[l], kv[l0 + l].k, kv_rows, HD)) != DDL_OK ||
          (st = encode_kv_map(&P.vmap[l], kv[l0 + l].v, kv_rows, HD)) != DDL_OK)
        return st;
    }
    const size_t need_trace = (size_t)nL * NSTAGE * C * TRACE_WORDS * 8;
    P.trace = (g_trace && g_trace_bytes >= need_trace && L <= MAX_LAYERS) ? g_trace : nullptr;
    if (l0 > 0 && (e = cudaMemsetAsync(ws + w.xmax, 0, (size_t)(w.gpart - w.xmax), cs)) != cudaSuccess)
      return cuda_status(e);  // maxima are per launch (its first layer finds its own)
    if (l0 > 0 && (e = cudaMemsetAsync(ws + w.gpart, 0xFF, (size_t)(w.apart - w.gpart), cs)) != cudaSuccess)
      return cuda_status(e);
    if (use_tc) {  // weight stages on the tensor cores, attention by the decode kernel
      TcLayer tl[MAX_LAYERS];
      for (int l = 0; l < nL; ++l)
        tl[l] = TcLayer{P.layers[l].packed, P.layers[l].norm1, P.layers[l].norm2, P.layers[l].kc, P.layers[l].vc};
      TcRun R;
      memset(&R, 0, sizeof R);
      R.D = P.D; R.Hq = P.Hq; R.Hkv = P.Hkv; R.hd = HD; R.dff = P.dff; R.B = B; R.GH = P.GH;
      R.wtype = wtype; R.C = C; R.eps = P.eps; R.pos = pos; R.s_max = s_max;
      memcpy(R.rope, P.rope, sizeof R.rope);
      R.posb = posv ? (const int32_t*)(ws + w.rope + (int64_t)B * 64 * 2 * 4) : nullptr;
      R.kv_bstride = P.kv_bstride;
      R.rope_b = posv ? (const float*)(ws + w.rope) : nullptr;
      R.ptab = P.ptab;
      R.pshift = P.pshift;
      R.pstride = P.pstride;
      make_geoms(*s, wtype, R.mg);
      R.layers = tl; R.L = nL; R.l0 = l0; R.final_last = P.final_last;
      R.resid_in = resid_in; R.x_bf16 = x_bf16; R.resid_out = resid_out; R.out_bf16 = out_bf16;
      R.status = P.ctrl + 1; R.wait_ns = g_wait_ns;
      R.q = P.q; R.attn = P.attn; R.y = P.y; R.a = P.a; R.Z = P.Z;
      tc_workspace_carve(*s, B, wtype, ws + w.tc, R);
      if ((st = tc_begin(R, stream))) return st;
      P.cooperative = 0;
      P.trace = nullptr;
      for (int l = 0; l < nL; ++l) {
        if ((st = tc_stage(R, l, ST_QKV, stream))) return st;
        P.stage_begin = l * NSTAGE + ST_ATT;
        P.stage_end = P.stage_begin + 1;
        void* args[] = {&P};
        if ((e = launch_pdl(fn, dim3(C), dim3(NTHREADS_ALL), args, SM_TOTAL, cs)) != cudaSuccess)
          return cuda_status(e);
        for (int stg : {ST_WO, ST_GU, ST_DOWN})
          if ((st = tc_stage(R, l, stg, stream))) return st;
      }
    } else if (coop) {
      if (l0 > 0 && (e = cudaMemsetAsync(ws + w.ctrl, 0, 4, cs)) != cudaSuccess) return cuda_status(e);
      P.stage_begin = 0;
      P.stage_end = nL * NSTAGE;
      P.cooperative = 1;
      void* args[] = {&P};
      e = cudaLaunchCooperativeKernel(fn, dim3(C), dim3(NTHREADS_ALL), args, SM_TOTAL, cs);
      if (e != cudaSuccess) return cuda_status(e);
    } else {
      P.cooperative = 0;
      for (int sidx = 0; sidx < nL * NSTAGE; ++sidx) {
        P.stage_begin = sidx;
        P.stage_end = sidx + 1;
        if (P.trace) P.trace = g_trace + (size_t)sidx * C * TRACE_WORDS;
        void* args[] = {&P};
        e = cudaLaunchKernel(fn, dim3(C), dim3(NTHREADS_ALL), args, SM_TOTAL, cs);
        if (e != cudaSuccess) return cuda_status(e);
      }
    }
  }
  return DDL_OK;
}

}  // namespace ddl

using namespace ddl;

extern "C" size_t ddl_workspace_bytes(const ddl_shape* shape, int32_t B, int64_t s_max) {
  if (check_shape(shape) || B < 1 || B > TC_MAX_B || s_max < 1) return 0;
  DevInfo di;
  if (device_info(di)) return 0;
  MatGeom mg[4];
  WsLayout w;
  if (plan(shape, DDL_W_INT4, B, s_max, di.sms, mg, w)) return 0;
  WsLayout w2;
  MatGeom mg2[4];
  if (plan(shape, DDL_W_BF16, B, s_max, di.sms, mg2, w2)) return 0;
  return (size_t)(w.total > w2.total ? w.total : w2.total);
}

extern "C" int ddl_workspace_view(const ddl_shape* shape, int32_t B, int64_t s_max,
                                  ddl_ws_view* out) {
  int st = check_shape(shape);
  if (st) return st;
  if (!out || B < 1 || B > TC_MAX_B || s_max < 1) return DDL_ERR_ARG;
  DevInfo di;
  if ((st = device_info(di))) return st;
  MatGeom mg[4];
  WsLayout w;
  if ((st = plan(shape, DDL_W_INT4, B, s_max, di.sms, mg, w))) return st;
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

extern "C" int ddl_stack_decode_ragged(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layers,
                                       const ddl_kv* kv, int32_t L, int32_t B, const int64_t* pos,
                                       const float* resid_in, const uint16_t* x_bf16, float* resid_out,
                                       uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream) {
  if (!pos) return DDL_ERR_ARG;
  if (B < 1 || B > TC_MAX_B) return DDL_ERR_UNSUPPORTED;
  return decode(shape, wtype, layers, kv, L, B, 0, resid_in, x_bf16, resid_out, out_bf16, workspace, ws_bytes,
                stream, pos);
}

extern "C" int ddl_stack_prefill(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layers,
                                 const ddl_kv* kv, int32_t L, int32_t S, int64_t p0, const float* resid_in,
                                 const uint16_t* x_bf16, float* resid_out, uint16_t* out_bf16, void* workspace,
                                 size_t ws_bytes, void* stream) {
  if (S < 1 || S > TC_MAX_B) return DDL_ERR_UNSUPPORTED;
  if (p0 < 0) return DDL_ERR_POS;
  int64_t pos[TC_MAX_B];
  for (int i = 0; i < S; ++i) pos[i] = p0 + i;  // (the last must stay below s_max: checked with the others)
  return decode(shape, wtype, layers, kv, L, S, 0, resid_in, x_bf16, resid_out, out_bf16, workspace, ws_bytes,
                stream, pos, true);
}

// The paged pools as the contiguous-cache descriptors decode() checks (the
// pointers and one logical s_max = pages_per_seq * page_size), and the page
// table's description; DDL_ERR_ARG when an argument is out of range.
static int paged_views(const ddl_kv_pages* kv, int32_t L, int32_t per_seq, int32_t page_size,
                       std::vector<ddl_kv>& out, Paged& pg, const int32_t* table) {
  if (!kv || !table || L <= 0 || per_seq < 1) return DDL_ERR_ARG;
  if (page_size < 16 || page_size > (1 << 20) || (page_size & (page_size - 1))) return DDL_ERR_ARG;
  const int64_t pages = kv[0].pages;
  if (pages < 1) return DDL_ERR_ARG;
  out.resize(L);
  for (int l = 0; l < L; ++l) {
    if (kv[l].pages != pages) return DDL_ERR_ARG;
    out[l] = ddl_kv{kv[l].k, kv[l].v, (int64_t)per_seq * page_size};
  }
  pg = Paged{table, per_seq, page_size, pages};
  return DDL_OK;
}

extern "C" int ddl_stack_decode_paged(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layers,
                                      const ddl_kv_pages* kv, int32_t L, int32_t B, const int64_t* pos,
                                      const int32_t* page_table, int32_t pages_per_seq, int32_t page_size,
                                      const float* resid_in, const uint16_t* x_bf16, float* resid_out,
                                      uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream) {
  if (!pos) return DDL_ERR_ARG;
  if (B < 1 || B > TC_MAX_B) return DDL_ERR_UNSUPPORTED;
  std::vector<ddl_kv> views;
  Paged pg;
  int st = paged_views(kv, L, pages_per_seq, page_size, views, pg, page_table);
  if (st) return st;
  return decode(shape, wtype, layers, views.data(), L, B, 0, resid_in, x_bf16, resid_out, out_bf16, workspace,
                ws_bytes, stream, pos, false, &pg);
}

extern "C" int ddl_stack_prefill_paged(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layers,
                                       const ddl_kv_pages* kv, int32_t L, int32_t S, int64_t p0,
                                       const int32_t* page_table, int32_t pages_per_seq, int32_t page_size,
                                       const float* resid_in, const uint16_t* x_bf16, float* resid_out,
                                       uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream) {
  if (S < 1 || S > TC_MAX_B) return DDL_ERR_UNSUPPORTED;
  if (p0 < 0) return DDL_ERR_POS;
  std::vector<ddl_kv> views;
  Paged pg;
  int st = paged_views(kv, L, pages_per_seq, page_size, views, pg, page_table);
  if (st) return st;
  int64_t pos[TC_MAX_B];
  for (int i = 0; i < S; ++i) pos[i] = p0 + i;
  return decode(shape, wtype, layers, views.data(), L, S, 0, resid_in, x_bf16, resid_out, out_bf16, workspace,
                ws_bytes, stream, pos, true, &pg);
}

extern "C" int ddl_set_launch_mode(int32_t mode) {
  if (mode != 0 && mode != 1) return DDL_ERR_ARG;
  g_launch_mode = mode;
  return DDL_OK;
}

extern "C" int ddl_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns = ns ? ns : WAIT_LIMIT_NS;
  return DDL_OK;
}

extern "C" int ddl_test_hold_barrier(int32_t stage) {
  if (stage < -1) return DDL_ERR_ARG;
  g_hold_stage = stage;
  return DDL_OK;
}

extern "C" int ddl_set_trace(void* device_buf, size_t bytes) {
  g_trace = (uint64_t*)device_buf;
  g_trace_bytes = device_buf ? bytes : 0;
  return DDL_OK;
}

extern "C" int ddl_read_device_status(const void* workspace, const ddl_shape* shape, int32_t B,
                                      int64_t s_max, int32_t* status_out, void* stream) {
  if (!status_out) return DDL_ERR_ARG;
  ddl_ws_view v;
  int st = ddl_workspace_view(shape, B, s_max, &v);
  if (st) return st;
  if (!workspace) {  // the static scratch of ddl_stack_decode_noalloc
    void* p = nullptr;
    if ((st = noalloc_scratch(&p)) != DDL_OK) return st;
    workspace = p;
  }
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
