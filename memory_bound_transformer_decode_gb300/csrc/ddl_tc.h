// ddl_tc.h -- the batched decode path on the 5th-generation (tcgen05) tensor
// cores: what the host runtime of ddl_decode.cu hands to it.
//
// At batch >= TC_MIN_B (INT4 weights) or > NARROW_B (bf16 weights) each layer
// runs as: QKV GEMM -> QKV epilogue (RMSNorm factor, RoPE, q, bf16 K/V append)
// -> attention (the decode kernel's attention stage, one launch) -> the
// attention output to tensor-core operands -> Wo GEMM -> Wo epilogue
// (residual, operands of gate/up) -> gate/up GEMM -> epilogue (SwiGLU,
// operands of down) -> down GEMM -> down epilogue (residual, operands of the
// next layer's QKV).
//
// Numerics.  A (weights) is fp16 holding code * scale exactly: |code| <= 7 is
// 3 bits and the bf16 scale 8, so the product has at most 11 significant bits
// (exact for scales in [2^-17, 9357]; bf16 weights are converted to fp16,
// exact for |w| >= 2^-17).  B (activations) is two fp16 limbs per value at
// the fixed scale 2^-8 (v = 256 (l0 + l1), l0 the fp16 rounding of v / 256,
// l1 that of the remainder): ~22 significant bits for |v| >= 32, an absolute
// 2^-17 below, |v| < 2^24, with no per-vector scale, so the producing
// epilogue writes them directly.  Products accumulate in fp32 in tensor
// memory; split-K partials are summed in a fixed order.
#pragma once
#include <stdint.h>

#include "../../include/ddl.h"
#include "ddl_plan.h"

namespace ddl {

constexpr int TC_MIN_B = 16;   // INT4 weights use the tensor-core path from this batch on
constexpr int TC_MAX_B = 64;   // largest batch of the library
constexpr int TC_EPI_CTAS = 304;
constexpr int TC_MAX_SPLIT = 8;

// Padded B-operand columns: two limbs per sequence, a multiple of 16.
inline int tc_ncols(int B) { return (2 * B + 15) & ~15; }

struct TcLayer {
  const uint8_t* packed;
  const uint16_t* norm1;
  const uint16_t* norm2;
  uint16_t* kc;
  uint16_t* vc;
};

// Everything one decode call of the tensor-core path needs (host side).
struct TcRun {
  int32_t D, Hq, Hkv, hd, dff, B, GH, wtype, C;
  float eps;
  int64_t pos, s_max;
  float rope[64][2];
  const int32_t* posb;           // ragged positions (device, [B]) or NULL: every sequence at pos
  const float* rope_b;           // [B][64][2] RoPE table of posb (device)
  int64_t kv_bstride;            // cache rows from sequence b to b + 1 (0: one shared cache)
  const int32_t* ptab;           // paged caches: page table (device), else NULL
  int32_t pshift, pstride;       // log2 page size, page-table entries per sequence (0: row 0 for all)
  MatGeom mg[4];                 // stream geometry (offsets into a packed layer)
  const TcLayer* layers;         // host array of this launch's layers
  int32_t L;                     // layers of this launch
  int32_t l0, final_last;        // global index of the first; its last is the stack's last
  const float* resid_in;         // layer-0 input (fp32) or NULL
  const uint16_t* x_bf16;        // layer-0 input (bf16) when resid_in is NULL
  float* resid_out;
  uint16_t* out_bf16;
  uint32_t* status;
  uint64_t wait_ns;
  // workspace
  float *q, *attn, *y, *a, *Z;   // Z: [2][B][D] residual ping-pong (as the decode kernel's)
  float* part;                   // split-K partials
  uint8_t* xl;                   // B-operand limb images of the next GEMM's input
  float* ss;                     // [2][TC_EPI_CTAS][B] partial sums of squares (QKV input, gate/up input)
  float* rfac;                   // [2][B] RMSNorm factors of those inputs (from ss, by the stage's GEMM)
};

// Workspace bytes of the path (beyond the decode kernel's own layout).
int64_t tc_workspace_bytes(const ddl_shape& s, int B, int wtype);
void tc_workspace_carve(const ddl_shape& s, int B, int wtype, uint8_t* base, TcRun& R);

// Before the first layer of a call: zero the limb images (padding columns)
// and, for the stack's first layer, turn its input into the QKV operands.
int tc_begin(const TcRun& R, void* stream);
// One weight stage (QKV, WO, GU or DOWN) of launch-local layer `layer`:
// operands -> GEMM -> epilogue.  For WO the attention output is converted
// first.
int tc_stage(const TcRun& R, int layer, int st, void* stream);

}  // namespace ddl
