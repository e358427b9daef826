// ddl_internal.h -- host-side helpers shared by the library's translation units:
// argument validation, CUDA error capture and the packed-layer geometry.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "../../include/ddl.h"
#include "ddl_plan.h"

namespace ddl {

void set_cuda_error(cudaError_t e);  // records cudaGetErrorString(e) for ddl_last_cuda_error
int noalloc_scratch(void** out);     // device address of ddl_stack_decode_noalloc's static scratch

inline int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DDL_OK;
  set_cuda_error(e);
  return DDL_ERR_CUDA;
}

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Shape rules of ddl.h.
inline int check_shape(const ddl_shape* s) {
  if (!s) return DDL_ERR_ARG;
  if (s->D <= 0 || s->H_q <= 0 || s->H_kv <= 0 || s->d_ff <= 0) return DDL_ERR_SHAPE;
  if (s->head_dim != 64 && s->head_dim != 128) return DDL_ERR_SHAPE;
  if (s->H_q % s->H_kv != 0 || s->H_q / s->H_kv > MAX_GH) return DDL_ERR_SHAPE;
  if (s->D % 64 || s->d_ff % 64 || (s->H_q * s->head_dim) % 64) return DDL_ERR_SHAPE;
  if (!(s->eps >= 0.f) || !(s->rope_base > 0.0)) return DDL_ERR_SHAPE;
  return DDL_OK;
}

inline int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// Geometry of the four streamed matrices of one layer (independent of the
// grid), and the byte size of a packed layer.
inline int64_t make_geoms(const ddl_shape& s, int wtype, MatGeom mg[4]) {
  const int32_t Nq = s.H_q * s.head_dim, Nkv = s.H_kv * s.head_dim;
  const int32_t dims[4][2] = {{Nq + 2 * Nkv, s.D}, {s.D, Nq}, {2 * s.d_ff, s.D}, {s.D, s.d_ff}};
  int64_t off = 0;
  for (int k = 0; k < 4; ++k) {
    MatGeom& m = mg[k];
    memset(&m, 0, sizeof m);
    m.N = dims[k][0];
    m.K = dims[k][1];
    m.NT = m.N / 16;
    m.G = m.K / DDL_GROUP;
    m.Gc = m.G < GC ? m.G : GC;
    m.Sk = (m.G + m.Gc - 1) / m.Gc;
    m.T = (int64_t)m.NT * m.G;
    m.woff = off;  // INT4: one stream of blocks, each its codes then its scales (one copy per slot)
    off = align256(off + m.T * (wtype == DDL_W_INT4 ? QBLK_BYTES : BF16_BLK_BYTES));
    m.soff = wtype == DDL_W_INT4 ? m.woff + BLK_BYTES : off;
    // the INT4 slot loop is bound by instruction issue, which the producer
    // warp shares with consumer warps 0 and 4; bf16 weights' streams wait on
    // memory, so their warps take equal shares
    m.even = wtype == DDL_W_BF16;
  }
  return off;
}

// Panels of a matrix for batch B on C CTAs (see ddl_plan.h): at most
// XF_CHUNKS / B k-chunks per panel, near-equal chunk counts, CTAs in
// proportion to blocks (at least one each); then J, the largest number of
// warps sharing a (tile, panel).  Returns false if the grid is too small.
inline bool make_panels(MatGeom& m, int B, int C) {
  // narrow batches: 2B fp16 columns per group; wider ones: 8 per n-tile of
  // ceil(B / 8) (fp16 without the low part), 4 x 256 bytes each
  int ch = B <= NARROW_B ? XF_CHUNKS / B : XF_CHUNKS / (4 * ((B + 7) / 8));
  if (ch < 1) ch = 1;
  int NP = (m.Sk + ch - 1) / ch;
  if (NP > MAXP || NP > C) return false;
  m.NP = NP;
  for (int p = 0; p <= NP; ++p) m.pk[p] = (int16_t)((int64_t)m.Sk * p / NP);
  int64_t acc = 0;
  m.pc[0] = 0;
  for (int p = 0; p < NP; ++p) {
    acc += panel_blocks(m, p);
    int c = (int)((acc * C + m.T / 2) / m.T);
    if (c < m.pc[p] + 1) c = m.pc[p] + 1;
    if (c > C - (NP - 1 - p)) c = C - (NP - 1 - p);
    m.pc[p + 1] = (int16_t)c;
  }
  m.pc[NP] = (int16_t)C;
  uint32_t J = 1;
  for (int p = 0; p < NP; ++p) {
    const uint32_t Gp = panel_groups(m, p);
    for (int T = 0; T < m.NT; ++T) {
      const uint32_t n = work_owner(m, p, (uint32_t)(T + 1) * Gp - 1, NW) -
                         work_owner(m, p, (uint32_t)T * Gp, NW) + 1;
      if (n > J) J = n;
    }
  }
  m.J = (int32_t)J;
  // a warp owns the split tiles whose first panel-0 block it holds; with more
  // than two it would wait for other contributors in mid-stream
  int maxown = 0;
  const uint32_t Gp0 = panel_groups(m, 0);
  for (int v = 0; v < (m.pc[1] - m.pc[0]) * NW; ++v) {
    uint32_t lo, hi;
    warp_work(m, 0, v / NW, v % NW, NW, lo, hi);
    int own = 0;
    for (uint32_t T = (lo + Gp0 - 1) / Gp0; T * Gp0 < hi; ++T)
      if (m.NP > 1 || (T + 1) * Gp0 > hi) ++own;
    if (own > maxown) maxown = own;
  }
  m.own_ok = maxown <= 2 && NP * (int)J <= 32;  // owners track a tile's slots in a 32-bit mask
  return true;
}

// A kernel launch that may overlap the previous kernel of the stream
// (programmatic dependent launch): its blocks may start while that kernel
// finishes, so the kernel waits (griddepcontrol.wait) before it reads what
// that kernel writes or writes what it reads.
inline cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, void** args, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace ddl
