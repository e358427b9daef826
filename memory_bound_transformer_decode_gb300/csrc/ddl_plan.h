// ddl_plan.h -- geometry of the packed weight streams and of the work split,
// shared by the host runtime and the kernels.
//
// Weight stream.  Each matrix W [N][K] (y = W x) is cut into 16-row tiles and
// 64-wide groups along K (the INT4 scale group).  One (tile, group) "block" is
// 512 bytes of 4-bit codes laid out in the register order of one
// m16n8k16 tensor-core A fragment per 16 columns: lane (g, t) = (lane/4,
// lane%4) owns 16 bytes = four 32-bit words, word j covering columns
// 16j..16j+15 of rows g and g+8.  Within a word the eight nibbles are
//   bits  0- 3: row g,   k 2t      bits 16-19: row g,   k 2t+1
//   bits  4- 7: row g+8, k 2t      bits 20-23: row g+8, k 2t+1
//   bits  8-11: row g,   k 2t+8    bits 24-27: row g,   k 2t+9
//   bits 12-15: row g+8, k 2t+8    bits 28-31: row g+8, k 2t+9
// (codes stay 4-bit two's complement, as in the canonical format).  The 16
// bf16 scales of a block follow in a separate stream, 8 words of
// (scale of row g | scale of row g+8 << 16).
// Blocks are ordered (k-chunk, tile, group-in-chunk) with k-chunks of GC=32
// groups (2048 columns; the last chunk may be shorter), so that a CTA's
// contiguous share of the stream touches at most two chunks of x.
//
// Row order inside tiles (the "row map"): QKV tiles pair row i of a head with
// row i + hd/2 (the two halves RoPE rotates together); gate/up tiles pair gate
// row j (rows 0-7) with up row j (rows 8-15); Wo and down tiles are 16
// consecutive rows.
//
// Work split: see panel_of_cta / warp_work below.  A tile covered by more
// than one warp is finished by the last warp that contributes to it (an
// atomic counter per tile), which sums the partial results in a fixed order:
// results do not depend on timing.
#pragma once
#include <cuda.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define DDL_HD __host__ __device__ __forceinline__
#else
#define DDL_HD inline
#endif

namespace ddl {

constexpr int NW = 8;                 // consumer warps per CTA (each consumes its own ring)
constexpr int NTHREADS = NW * 32;     // consumer threads
// A CTA is three warpgroups: the consumer warps (warpgroups 0 and 1) and a
// third whose first warp fills every consumer warp's ring (its other three
// warps leave at once).  setmaxnreg moves registers from the producer
// warpgroup to the consumers: PRODUCER_REGS * 128 + CONSUMER_REGS * 256 must
// not exceed the launch's 384 threads x 168 registers.
constexpr int NTHREADS_ALL = 384;
constexpr int PRODUCER_REGS = 40;
constexpr int CONSUMER_REGS = 232;
constexpr int PRODUCER_NAP_NS = 100;  // the producer's pause after a round with nothing to issue
static_assert(PRODUCER_REGS * 128 + CONSUMER_REGS * 256 <= NTHREADS_ALL * 168, "register split");
constexpr int DEPTH = 3;              // ring slots per warp
constexpr int SLOT_BYTES = 4608;      // 8 INT4 blocks with their scales, or 16 KV rows (512-byte aligned)
constexpr int BLK_BYTES = 512;        // one INT4 block: 16 rows x 64 columns
constexpr int SCL_BYTES = 32;         // scales of one block
constexpr int QBLK_BYTES = BLK_BYTES + SCL_BYTES;  // an INT4 block's codes followed by its scales
constexpr int BLKS_PER_SLOT = 8;
constexpr int BF16_BLK_BYTES = 2048;  // one bf16 block: 16 rows x 64 columns
constexpr int BF16_BLKS_PER_SLOT = 2;
constexpr int GC = 32;                // groups per k-chunk
constexpr int MAX_LAYERS = 96;        // layers per launch (longer stacks use several launches)
constexpr int MAX_B = 16;             // sequences of a batch
constexpr int NARROW_B = 4;           // up to this batch x is carried as fp16 hi/lo columns
// Up to this batch (INT4) a weight stage's producer writes the next stage's
// input as a fragment image that the next prologue bulk-copies into place; at
// 3 and 4 sequences the image's bytes (4 per element per sequence) cost more
// than the in-place conversion they replace (measured on one GB300: batch 2
// 286 vs 263 tokens/s with and without, batch 4 336 vs 347).
constexpr int IMG_MAX_B = 2;
constexpr int MAX_GH = 8;             // query heads per KV head
constexpr int NSTAGE = 5;
constexpr int MAXP = 16;              // k-chunk panels per matrix
constexpr int XF_CHUNKS = 8;          // k-chunks of x one CTA can stage at batch 1 (x batch size <= 8)
constexpr int TRACE_WORDS = 2 * NW + 16;  // per (stage, CTA) in the optional trace

// Floats of one attention softmax record (o[GH][hd], m[GH], l[GH]), padded
// to 16 bytes so that records can be read as float4.
DDL_HD int att_rec_floats(int GH, int hd) { return (GH * (hd + 2) + 3) & ~3; }

enum Stage { ST_QKV = 0, ST_ATT = 1, ST_WO = 2, ST_GU = 3, ST_DOWN = 4 };
enum MatKind { MK_QKV = 0, MK_WO = 1, MK_GU = 2, MK_DOWN = 3 };

DDL_HD int stage_mat(int st) {
  return st == ST_QKV ? MK_QKV : st == ST_WO ? MK_WO : st == ST_GU ? MK_GU : st == ST_DOWN ? MK_DOWN : -1;
}

struct MatGeom {
  int32_t N, K;       // rows of the (combined) matrix, input dimension
  int32_t NT, G;      // 16-row tiles, 64-column groups per row
  int32_t Gc, Sk;     // groups per full k-chunk, number of k-chunks
  int32_t J;          // partial slots per (tile, panel)
  int32_t NP;         // panels: k-chunks pk[p]..pk[p+1]-1, worked by CTAs pc[p]..pc[p+1]-1
  int32_t own_ok;     // split tiles may be finished by their owners: no warp owns more than two
  int32_t even;       // equal warp shares (bf16 weights: data-bound streams), else 15 : 16 for warps 0 and 4
  int64_t T;          // blocks
  int64_t woff, soff; // packed layer: INT4 block b's codes at woff + b * QBLK_BYTES, its scales at
                      // soff + b * QBLK_BYTES (soff = woff + BLK_BYTES); bf16 block b at woff + b * 2048
  int16_t pk[MAXP + 1];
  int16_t pc[MAXP + 1];
};

DDL_HD int32_t chunk_groups(const MatGeom& m, int kc) {
  return kc == m.Sk - 1 ? m.G - (m.Sk - 1) * m.Gc : m.Gc;
}
DDL_HD int64_t chunk_start(const MatGeom& m, int kc) { return (int64_t)kc * m.NT * m.Gc; }
DDL_HD void block_coord(const MatGeom& m, int64_t b, int& kc, int& T, int& gi) {
  int64_t per = (int64_t)m.NT * m.Gc;
  kc = (int)(b / per);
  if (kc > m.Sk - 1) kc = m.Sk - 1;
  int64_t rem = b - chunk_start(m, kc);
  int gk = chunk_groups(m, kc);
  T = (int)(rem / gk);
  gi = (int)(rem % gk);
}
DDL_HD int64_t unit_start(const MatGeom& m, int kc, int T) {
  return chunk_start(m, kc) + (int64_t)T * chunk_groups(m, kc);
}
// Contiguous split of [0, total) into `parts` ranges: range i = [lo(i), lo(i+1)).
DDL_HD int64_t range_lo(int64_t total, int64_t parts, int64_t i) { return total * i / parts; }
// The part owning item b (total > 0).
DDL_HD int64_t owner_of(int64_t total, int64_t parts, int64_t b) {
  return ((b + 1) * parts - 1) / total;
}

// 32-bit forms for the kernels (the host checks T * W < 2^32).
DDL_HD uint32_t owner32(uint32_t total, uint32_t parts, uint32_t b) {
  return ((b + 1) * parts - 1) / total;
}
DDL_HD uint32_t lo32(uint32_t total, uint32_t parts, uint32_t i) { return total * i / parts; }
DDL_HD uint32_t unit_start32(const MatGeom& m, int kc, int T) {
  return (uint32_t)kc * (uint32_t)m.NT * (uint32_t)m.Gc + (uint32_t)T * (uint32_t)chunk_groups(m, kc);
}

// Work split.  The k-chunks are grouped into panels of at most as many
// chunks as one CTA can stage; panel p gets CTAs pc[p]..pc[p+1]-1 in
// proportion to its blocks.  Inside a panel the work order is tile-major
// (tile, k-chunk, group), so a warp accumulates a whole tile across the
// panel's chunks in registers; within a panel the CTAs, and within a CTA the
// warps, take contiguous ranges of that order.  Only tiles split between
// warps or panels leave partials: slot (tile, panel, j) for the j-th warp
// (in panel order) owning blocks of the tile; each contributor adds its block
// count to the tile's counter and the one that brings it to G finishes it.
DDL_HD int panel_of_cta(const MatGeom& m, int c) {
  int p = 0;
  while (p + 1 < m.NP && c >= m.pc[p + 1]) ++p;
  return p;
}
DDL_HD uint32_t panel_groups(const MatGeom& m, int p) {
  const int k0 = m.pk[p], k1 = m.pk[p + 1];
  return (uint32_t)((k1 - k0) * m.Gc - (k1 == m.Sk ? m.Sk * m.Gc - m.G : 0));
}
DDL_HD uint32_t panel_blocks(const MatGeom& m, int p) { return (uint32_t)m.NT * panel_groups(m, p); }
// Range of panel work indices of warp w (0..NW-1) of panel-local CTA cl.
// Inside a CTA's range of R blocks the eight consumer warps take shares in
// proportion 15 : 16 for the two warps that share their scheduler with the
// producer warp (warps 0 and 4) and the others: that scheduler issues the
// producer's instructions too, and its consumer warps measured ~6 % slower.
DDL_HD uint32_t warp_lo(uint32_t R, int nw, int w, bool even = false) {
  if (nw != 8 || even) return lo32(R, (uint32_t)nw, (uint32_t)w);
  const uint32_t cum = 16u * (uint32_t)w - (uint32_t)((w + 3) / 4);  // sum of the shares of warps < w
  return (uint32_t)((uint64_t)R * cum / 126u);
}
DDL_HD void warp_work(const MatGeom& m, int p, int cl, int w, int nw, uint32_t& lo, uint32_t& hi) {
  const uint32_t Tp = panel_blocks(m, p), Cp = (uint32_t)(m.pc[p + 1] - m.pc[p]);
  const uint32_t clo = lo32(Tp, Cp, cl), R = lo32(Tp, Cp, cl + 1) - clo;
  lo = clo + warp_lo(R, nw, w, m.even);
  hi = clo + warp_lo(R, nw, w + 1, m.even);
}
// Panel-local warp index (cl * nw + w) owning panel work index i.
DDL_HD uint32_t work_owner(const MatGeom& m, int p, uint32_t i, int nw) {
  const uint32_t Tp = panel_blocks(m, p), Cp = (uint32_t)(m.pc[p + 1] - m.pc[p]);
  const uint32_t cl = owner32(Tp, Cp, i), clo = lo32(Tp, Cp, cl), R = lo32(Tp, Cp, cl + 1) - clo;
  uint32_t w = 0;
  while ((int)w + 1 < nw && warp_lo(R, nw, (int)w + 1, m.even) <= i - clo) ++w;
  return cl * nw + w;
}
DDL_HD bool warp_empty(const MatGeom& m, int p, uint32_t v, int nw) {
  uint32_t lo, hi;
  warp_work(m, p, (int)(v / nw), (int)(v % nw), nw, lo, hi);
  return lo == hi;
}
// (tile, k-chunk, group) of panel work index i.
DDL_HD void work_coord(const MatGeom& m, int p, uint32_t i, int& T, int& kc, int& gi) {
  const uint32_t Gp = panel_groups(m, p);
  T = (int)(i / Gp);
  const uint32_t r = i - (uint32_t)T * Gp;
  kc = m.pk[p] + (int)(r / (uint32_t)m.Gc);
  gi = (int)(r - (uint32_t)(kc - m.pk[p]) * (uint32_t)m.Gc);
}

// Row of the combined matrix held by row r (0..15) of tile T.
DDL_HD int32_t tile_row(int kind, int T, int r, int hd) {
  if (kind == MK_QKV) {
    int tph = hd / 16, head = T / tph, mm = T % tph;
    return head * hd + (r < 8 ? 8 * mm + r : 8 * mm + (r - 8) + hd / 2);
  }
  if (kind == MK_GU) return r < 8 ? 8 * T + r : 8 * T + (r - 8);  // gate row / up row
  return 16 * T + r;
}

struct LayerDev {
  const uint8_t* packed;
  const uint16_t* norm1;
  const uint16_t* norm2;
  uint16_t* kc;
  uint16_t* vc;
};

struct Params {
  int32_t D, Hq, Hkv, hd, dff, B, GH;  // GH = Hq / Hkv
  float eps;
  int32_t wtype;
  double rope_base;
  int64_t pos, s_max;
  int32_t L;            // layers in this launch
  int32_t l0;           // global index of this launch's first layer
  int32_t final_last;   // this launch's last layer is the stack's last
  int32_t stage_begin, stage_end;  // flattened (layer * NSTAGE + stage) range
  int32_t cooperative;
  int32_t nt_att;       // 16-key tiles per sequence
  int32_t J_att;        // attention partial slots per sequence
  int32_t hold_stage;   // test hook: the grid barrier before this flattened stage of the step waits for ever (-1: none)
  uint64_t wait_ns;     // limit of every bounded wait
  float rope[64][2];    // cos, sin of pos * base^(-2i/hd), i < hd/2 (computed in fp64 on the host)
  MatGeom mg[4];
  const float* resid_in;
  const uint16_t* x_bf16;
  float* resid_out;
  uint16_t* out_bf16;
  uint32_t* ctrl;       // [0] grid barrier counter, [1] status word
  uint32_t* cnt;        // per-tile arrival counters
  uint32_t* seqcnt;     // per-sequence arrival counters of the attention merge
  uint32_t* xmax;       // [layer][stage][MAX_B] bits of max |x * norm weight| of a stage's input, from its producer
  float* gpart;         // GEMV partials: [tile][panel][J][32 lanes][2]
  float* apart;         // attention partials: [seq][J_att][GH*(hd+2)]
  float* Z;             // [2][B][D] residual ping-pong between layers
  float* q;             // [B][Hq*hd]
  float* attn;          // [B][Hq*hd]
  float* y;             // [B][D]
  float* a;             // [B][dff]
  uint8_t* ximg[2];     // INT4, B <= 4: fp16 fragment images of the next weight stage's input, by stage parity (or NULL)
  int32_t ragged;       // sequences at their own positions: posb, rope_b (else every sequence at pos, rope)
  int32_t posb[64];     // position of sequence b (ragged)
  const float* rope_b;  // [B][64][2] cos, sin of posb[b] * base^(-2i/hd) (ragged)
  int64_t kv_bstride;   // cache rows from sequence b to b + 1: H_kv * s_max, or 0 when the rows share one cache (prefill)
  int32_t p0;           // prefill: the first prompt position (rows p0 .. are written in this step), else -1
  // paged caches (pshift > 0): slot t of sequence b sits in page ptab[b * pstride + (t >> pshift)],
  // row t & (2^pshift - 1); the K/V views are then [pages * H_kv * 2^pshift rows][hd]
  const int32_t* ptab;  // device copy of the page table (workspace)
  int32_t pshift;       // log2 of the page size (0: contiguous caches)
  int32_t pstride;      // page-table entries per sequence (0: every row reads row 0, prefill)
  uint64_t* trace;      // optional: per stage, CTA: start, prologue end, NW warp ends, end, 4 prologue steps (ns)
  LayerDev layers[MAX_LAYERS];
  // 2-D views [B * H_kv * s_max rows][hd] of each layer's K and V caches for
  // TMA tensor copies of 16 rows x 64 columns with the 128-byte swizzle
  CUtensorMap kmap[MAX_LAYERS];
  CUtensorMap vmap[MAX_LAYERS];
};

}  // namespace ddl
