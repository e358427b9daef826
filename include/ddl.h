/*
 * ddl.h -- C ABI of the GB300 (sm_103a) batch-B INT4 GQA decode step.
 *
 * The library computes one autoregressive decode step of a stack of GQA
 * transformer decoder layers ("把基础打牢" primer, §1.1 block and §1.2
 * decode_step): per layer
 *     h = rmsnorm(x, norm1);  q, k, v = h Wq, h Wk, h Wv;  RoPE on q and k;
 *     append bf16(k), bf16(v) to the KV cache at slot pos;
 *     attn = softmax(q K^T / sqrt(hd)) V over slots 0..pos, K/V head
 *            floor(h / (H_q / H_kv)) shared by its query group;
 *     y = x + attn Wo;  z = y + (silu(h2 Wg) * (h2 Wu)) Wd,  h2 = rmsnorm(y, norm2)
 * with the 4-bit weights expanded to floating point only in registers
 * (Unsloth/Qwen-27B article, §二.3) and RMSNorm, RoPE, the KV append,
 * SwiGLU and the residual adds fused into the weight-streaming kernels
 * (same article §二.1; roofline reply, §三 lever 1).
 *
 * Conventions (every entry point):
 *  - Pointers marked "device" are CUDA device pointers owned by the caller;
 *    the library never frees them and allocates no device memory on the
 *    decode path.  Pointers marked "host" are ordinary host memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous on it unless stated otherwise.
 *  - Return value: DDL_OK (0) or a ddl_status code; nothing throws, nothing
 *    traps.  Argument errors are found on the host before any launch.  A
 *    device-side wait that gives up (DDL_ERR_TIMEOUT) is recorded in the
 *    workspace and read back with ddl_read_device_status().
 *  - bf16 tensors are passed as uint16_t bit patterns.
 *  - All device pointers must be 16-byte aligned (DDL_ERR_ALIGN otherwise).
 */
#ifndef DDL_H
#define DDL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DDL_GROUP 64      /* INT4 scale group along the input dimension K */
#define DDL_MAX_BATCH 64  /* sequences per step */
#define DDL_MAX_GROUP_HEADS 8 /* H_q / H_kv */

typedef enum {
    DDL_OK = 0,
    DDL_ERR_SHAPE = 1,       /* a dimension is not supported (see ddl_shape) */
    DDL_ERR_POS = 2,         /* pos < 0 or pos >= s_max */
    DDL_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned */
    DDL_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than ddl_workspace_bytes() */
    DDL_ERR_UNSUPPORTED = 5, /* weight type / batch / layer count not supported */
    DDL_ERR_CUDA = 6,        /* a CUDA runtime call failed (see ddl_last_cuda_error) */
    DDL_ERR_TIMEOUT = 7,     /* a bounded device wait gave up (device status word) */
    DDL_ERR_ARG = 8          /* NULL pointer or negative size */
} ddl_status;

/* Layer shape.  Supported: D, d_ff, H_q*head_dim multiples of 64;
 * head_dim in {64, 128}; H_q % H_kv == 0 with H_q/H_kv <= 8; eps >= 0. */
typedef struct {
    int32_t D;          /* model width */
    int32_t H_q;        /* query heads */
    int32_t H_kv;       /* key/value heads */
    int32_t head_dim;   /* hd */
    int32_t d_ff;       /* SwiGLU hidden width */
    float eps;          /* RMSNorm epsilon, inside the square root */
    double rope_base;   /* RoPE base: angle of pair i at position p is p * base^(-2i/hd) */
} ddl_shape;

typedef enum { DDL_W_INT4 = 0, DDL_W_BF16 = 1 } ddl_wtype;

/* One weight matrix W [N][K] (y = W x) in the canonical formats:
 *  INT4: q [N][K/2] uint8, two 4-bit two's-complement codes per byte, even k
 *        in the low nibble; scale [N][K/64] bf16.  W[n][k] = code * scale.
 *  BF16: w [N][K] bf16.
 * All device pointers. */
typedef struct {
    const uint8_t* q;
    const uint16_t* scale;
    const uint16_t* w;
} ddl_mat;

/* One layer's matrices in canonical format (input of ddl_pack_layer).
 * Shapes: wq [H_q*hd][D], wk/wv [H_kv*hd][D], wo [D][H_q*hd],
 * wg/wu [d_ff][D], wd [D][d_ff]. */
typedef struct {
    ddl_mat wq, wk, wv, wo, wg, wu, wd;
} ddl_layer_src;

/* One layer as the decode kernels read it.
 *  packed: device blob written by ddl_pack_layer (ddl_packed_layer_bytes).
 *  norm1, norm2: device bf16 [D] RMSNorm weights. */
typedef struct {
    const void* packed;
    const uint16_t* norm1;
    const uint16_t* norm2;
} ddl_layer_w;

/* One layer's KV cache: k and v each [B][H_kv][s_max][head_dim] bf16, device.
 * Slots 0..pos-1 hold the history; decode writes slot pos. */
typedef struct {
    uint16_t* k;
    uint16_t* v;
    int64_t s_max;
} ddl_kv;

/* One layer's paged KV cache: k and v each [pages][H_kv][page_size][head_dim]
 * bf16, device.  A sequence's slots live in pages named by its row of a page
 * table (ddl_stack_decode_paged); every layer uses the same page table. */
typedef struct {
    uint16_t* k;
    uint16_t* v;
    int64_t pages;
} ddl_kv_pages;

/* ------------------------------------------------------------ weights */

/* Symmetric INT4 quantization with group 64 along K and a bf16 scale per
 * group (4-bit storage expanded with its scale on arrival, Unsloth/Qwen-27B
 * article §二.3; format: symmetric, group 64, low nibble first):
 *     s = bf16_rne(max|w_group| / 7),  code = clamp(rne(w / s), -7, 7),
 *     all-zero group -> s = 0, codes 0.
 * w_bf16: device [N][K] bf16.  q_out: device [N][K/2].  scale_out: device
 * [N][K/64].  K must be a multiple of 64, N >= 1.  Bit-exact with the oracle. */
int ddl_quantize_int4(const uint16_t* w_bf16, int64_t N, int64_t K, uint8_t* q_out,
                      uint16_t* scale_out, void* stream);

/* Bytes of one packed layer for `shape` and weight type. */
size_t ddl_packed_layer_bytes(const ddl_shape* shape, ddl_wtype wtype);

/* Rearrange one layer's canonical matrices into the kernel-native stream
 * (a permutation of the same codes, scales or bf16 values: 16-row tiles in
 * tensor-core fragment order, RoPE pair rows and gate/up rows side by side,
 * the input dimension cut into chunks of 2048).  src: device canonical
 * matrices of `wtype`; packed_out: device, ddl_packed_layer_bytes() bytes. */
int ddl_pack_layer(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_src* src,
                   void* packed_out, void* stream);

/* ------------------------------------------------------------ KV cache */

/* Append one token's k and v for B sequences at slot pos (primer §1.2
 * append_to_kv_cache): K[b][g][pos][:] = k_new[b][g][:], same for V.
 * k_new, v_new: device [B][H_kv][head_dim] bf16.  Pure copy, bit-exact. */
int ddl_kv_append(const ddl_kv* kv, int32_t B, int32_t H_kv, int32_t head_dim, int64_t pos,
                  const uint16_t* k_new, const uint16_t* v_new, void* stream);

/* ------------------------------------------------------------ decode */

/* Device workspace bytes for a decode call with this shape, batch and
 * cache length (depends on the device's SM count; query on the device the
 * call will run on). */
size_t ddl_workspace_bytes(const ddl_shape* shape, int32_t B, int64_t s_max);

/* Where the per-stage results of the last layer of a call live inside the
 * workspace (byte offsets; fp32 arrays):
 *   q [B][H_q*hd] after RoPE, attn [B][H_q*hd], y [B][D], a [B][d_ff],
 *   and the device status word (int32). */
typedef struct {
    size_t q, attn, y, a, status;
} ddl_ws_view;
int ddl_workspace_view(const ddl_shape* shape, int32_t B, int64_t s_max, ddl_ws_view* out);

/* One decode step of one layer for B <= DDL_MAX_BATCH sequences, all at
 * position pos.  INT4 weights at B >= 16 and bf16 weights at B >= 5 run their
 * matrix products on the tcgen05 tensor cores (weights as fp16 code * scale,
 * exact for group scales in [2^-17, 9357]; bf16 weights converted to fp16,
 * exact for |w| >= 2^-17; activations as two fp16 limbs), smaller batches on
 * warp-level tensor-core MMAs inside one persistent kernel.  The step:
 * writes KV slot pos and attends over slots 0..pos (the caller keeps slots
 * < pos filled).  Input: resid_in [B][D] fp32, or x_bf16 [B][D] bf16 when
 * resid_in is NULL.  Output: resid_out [B][D] fp32 (may be NULL) and
 * out_bf16 [B][D] (may be NULL).  Outputs must not alias inputs.
 * workspace: device, >= ddl_workspace_bytes(shape, B, kv->s_max).
 * Calls sharing a workspace must be ordered on one stream. */
int ddl_layer_decode(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layer,
                     const ddl_kv* kv, int32_t B, int64_t pos, const float* resid_in,
                     const uint16_t* x_bf16, float* resid_out, uint16_t* out_bf16,
                     void* workspace, size_t ws_bytes, void* stream);

/* One decode step of an L-layer stack (primer §1.2 decode_step without the
 * embedding and sampling): layer l's output residual (fp32) is layer l+1's
 * input.  layers, kv: host arrays of L entries (device pointers inside);
 * every kv[l] has the same s_max.  Other arguments as ddl_layer_decode.
 * The whole stack runs as one persistent cooperative kernel (one CTA per
 * SM) when the device allows it, else one launch per fused stage. */
int ddl_stack_decode(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layers,
                     const ddl_kv* kv, int32_t L, int32_t B, int64_t pos,
                     const float* resid_in, const uint16_t* x_bf16, float* resid_out,
                     uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream);

/* ddl_stack_decode for sequences at their own positions (continuous
 * batching: sequences that joined at different times decode together; the
 * primer's §1.3 batching with a per-sequence history): sequence b writes KV
 * slot pos[b] of its own cache, attends over its slots 0..pos[b] and rotates
 * q, k by position pos[b].  pos: host array of B positions, each in
 * [0, s_max) (DDL_ERR_POS otherwise).  Slots past pos[b] may hold anything:
 * they are neither read into the result nor written.  Other arguments as
 * ddl_stack_decode; the workspace is sized by ddl_workspace_bytes. */
int ddl_stack_decode_ragged(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layers,
                            const ddl_kv* kv, int32_t L, int32_t B, const int64_t* pos,
                            const float* resid_in, const uint16_t* x_bf16, float* resid_out,
                            uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream);

/* Prefill of S <= DDL_MAX_BATCH prompt tokens of one sequence (primer §1.2:
 * the prompt goes through the layers and its K/V are kept in the cache) as
 * one batched step: row i is the token at position p0 + i; it writes slot
 * p0 + i of the sequence's cache and attends over slots 0..p0 + i, the
 * history and the prompt's rows before it (causal).  kv: the sequence's own
 * caches, each [1][H_kv][s_max][head_dim]; p0 + S <= s_max (DDL_ERR_POS).
 * x_bf16 / resid_in: [S][D] (row i the token at p0 + i); outputs [S][D].  A
 * longer prompt goes in chunks, p0 advancing by S each call.  The workspace
 * is sized by ddl_workspace_bytes(shape, S, s_max).  Other arguments as
 * ddl_stack_decode. */
int ddl_stack_prefill(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layers,
                      const ddl_kv* kv, int32_t L, int32_t S, int64_t p0, const float* resid_in,
                      const uint16_t* x_bf16, float* resid_out, uint16_t* out_bf16, void* workspace,
                      size_t ws_bytes, void* stream);

/* ddl_stack_decode_ragged on a paged KV cache (continuous batching, the
 * primer's §1.3, with each sequence's history in fixed-size pages, so that
 * sequences of any length share one pool without a contiguous region each):
 * slot t of sequence b lives in page page_table[b * pages_per_seq +
 * t / page_size] of every layer's pool, at row t % page_size.
 *  - kv: L pools, each [pages][H_kv][page_size][head_dim] bf16 (device), all
 *    with the same page count.
 *  - page_table: host int32 [B][pages_per_seq], copied to the workspace
 *    during the call (the caller may reuse it once the call returns).  Only
 *    the live entries (pages of slots 0..pos[b]) are read; each must lie in
 *    [0, pages), and the page that receives sequence b's new row must occur
 *    once among all live entries of the batch (no sequence reads a page
 *    being written, as with shared prefix pages) -- DDL_ERR_ARG otherwise.
 *  - page_size: a power of two in [16, 2^20] (DDL_ERR_ARG); pos[b] <
 *    pages_per_seq * page_size (DDL_ERR_POS); pages * H_kv * page_size <
 *    2^31 (DDL_ERR_UNSUPPORTED).
 *  - The workspace is sized by ddl_workspace_bytes(shape, B,
 *    pages_per_seq * page_size).  Other arguments as ddl_stack_decode_ragged. */
int ddl_stack_decode_paged(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layers,
                           const ddl_kv_pages* kv, int32_t L, int32_t B, const int64_t* pos,
                           const int32_t* page_table, int32_t pages_per_seq, int32_t page_size,
                           const float* resid_in, const uint16_t* x_bf16, float* resid_out,
                           uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream);

/* ddl_stack_prefill into a paged KV cache: the S prompt rows of one sequence
 * at positions p0..p0 + S - 1 write their K/V through the one page-table row
 * page_table[0 .. pages_per_seq) and attend causally over the slots before
 * them.  The pages receiving rows must each occur once among the live
 * entries (pages of slots 0..p0 + S - 1).  Other rules as
 * ddl_stack_decode_paged with B = 1; the workspace is sized by
 * ddl_workspace_bytes(shape, S, pages_per_seq * page_size). */
int ddl_stack_prefill_paged(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layers,
                            const ddl_kv_pages* kv, int32_t L, int32_t S, int64_t p0,
                            const int32_t* page_table, int32_t pages_per_seq, int32_t page_size,
                            const float* resid_in, const uint16_t* x_bf16, float* resid_out,
                            uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream);

/* Size of the library's own static scratch array (32 MiB), used only by
 * ddl_stack_decode_noalloc. */
#define DDL_NOALLOC_SCRATCH_BYTES (32u << 20)

/* ddl_stack_decode without a workspace argument, for callers that cannot
 * allocate device memory (a plugin whose host framework owns all device
 * memory and passes only inputs and outputs, or a loop that must not take
 * cudaMalloc's implicit device synchronization).  The pages have no
 * counterpart: this is an interface convenience, not part of the method.
 * Arguments and results are those of ddl_stack_decode.  The scratch is a
 * file-scope device array of DDL_NOALLOC_SCRATCH_BYTES that every GPU loading
 * the library keeps until process exit; the call allocates nothing.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - Returns DDL_ERR_WORKSPACE when the shape, batch and cache length need
 *    more scratch than DDL_NOALLOC_SCRATCH_BYTES (ddl_workspace_bytes tells).
 *  - All calls share the array and a call leaves its contents behind; calls
 *    that overlap on the GPU (other streams, other threads) race on it, so
 *    order them on one stream.
 *  - The device status word of the last call (DDL_OK or DDL_ERR_TIMEOUT) is
 *    read with ddl_read_device_status(NULL, ...). */
int ddl_stack_decode_noalloc(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_w* layers,
                             const ddl_kv* kv, int32_t L, int32_t B, int64_t pos,
                             const float* resid_in, const uint16_t* x_bf16, float* resid_out,
                             uint16_t* out_bf16, void* stream);

/* ------------------------------------------------------------ token step
 * The steps on either side of the layer stack in the primer's §1.2
 * decode step: the last token's embedding row before it, and after it a token
 * drawn from the logits of the last hidden state against the embedding table,
 * for a vocabulary of V entries (Unsloth/Qwen-27B article §三:
 * about 152 thousand, reduced chunk by chunk without forming the
 * distribution over the whole vocabulary). */

#define DDL_MAX_TOP_K 1024  /* largest k of top-k sampling */

/* Rows of the bf16 embedding table: x_out[b] = table[tokens[b]].
 * table: device [V][D] bf16 (D a multiple of 64).  tokens: device int32 [B],
 * B <= DDL_MAX_BATCH.  x_out: device [B][D] bf16 (the x_bf16 input of
 * ddl_stack_decode).  A token id outside [0, V) gives a zero row and, when
 * bad_out (device int32, may be NULL) is given, sets *bad_out to 1 (the call
 * never clears it). */
int ddl_embed(const uint16_t* table, int64_t V, int32_t D, const int32_t* tokens, int32_t B,
              uint16_t* x_out, int32_t* bad_out, void* stream);

/* Bytes of a packed output matrix [V][D] (0 if the arguments are invalid). */
size_t ddl_packed_head_bytes(int32_t D, int64_t V, ddl_wtype wtype);

/* Pack the output matrix (the tied embedding table: INT4 codes and scales
 * from ddl_quantize_int4, or the bf16 table) into the layout ddl_lm_head
 * streams: 16-row x 64-column blocks in the layers' block format, ordered
 * (16-row tile, group); rows past V in the last tile are zero.  Setup only. */
int ddl_pack_head(const ddl_mat* w, int32_t D, int64_t V, ddl_wtype wtype, void* packed_out,
                  void* stream);

/* Workspace bytes of ddl_lm_head for (D, V, B) on the current device. */
size_t ddl_head_workspace_bytes(int32_t D, int64_t V, int32_t B);

/* The LM head and the choice of the next token for B <= DDL_MAX_BATCH
 * sequences:  l = W h  with  h = rmsnorm(x, norm_f) when norm_f is given
 * (eps inside the square root, as the layers' RMSNorm), else h = x.
 *  x: device [B][D] fp32 (the stack's resid_out).  norm_f: device bf16 [D]
 *    or NULL.  head_packed: from ddl_pack_head.
 *  top_k <= 1: greedy, token_out[b] = the id of the largest logit (the
 *    lowest id among equal maxima).
 *  1 < top_k <= DDL_MAX_TOP_K: top-k sampling: the min(top_k, V) largest
 *    logits (equal logits at the boundary: lower ids first) in the order
 *    (logit descending, id ascending) with weights exp((l - l_max) / T),
 *    T = temperature > 0; token_out[b] is the first candidate whose
 *    cumulative weight exceeds u[b] * total (u: device fp32 [B] in [0, 1),
 *    drawn by the caller).
 *  logits_out: device fp32 [B][V] or NULL.  lse_out: device fp32 [B]
 *    (log sum_v exp(l_v)) or NULL.  token_out: device int32 [B].
 *  workspace: device, >= ddl_head_workspace_bytes(D, V, B).
 * Errors: DDL_ERR_ARG (NULL pointer, top_k < 0, temperature or u missing
 * for sampling), DDL_ERR_SHAPE (D not a multiple of 64), DDL_ERR_UNSUPPORTED
 * (B or top_k too large), DDL_ERR_ALIGN, DDL_ERR_WORKSPACE. */
int ddl_lm_head(int32_t D, int64_t V, ddl_wtype wtype, const void* head_packed, const uint16_t* norm_f,
                float eps, int32_t B, const float* x, int32_t top_k, float temperature, const float* u,
                int32_t* token_out, float* logits_out, float* lse_out, void* workspace, size_t ws_bytes,
                void* stream);

/* Launch mode of the decode calls: 0 = automatic (persistent cooperative
 * kernel when possible), 1 = one launch per fused stage. */
int ddl_set_launch_mode(int32_t mode);

/* Limit of every bounded wait inside the decode kernels (a wait for a TMA
 * copy, a grid barrier, another CTA's partial sums): a wait that gives up sets
 * the device status word to DDL_ERR_TIMEOUT and the kernel returns without
 * faulting; later calls on the same context work.  Applies to later calls;
 * ns = 0 restores the default of 2 s. */
int ddl_set_wait_limit_ns(uint64_t ns);

/* Test hook for the timeout path: when stage >= 0, the grid barrier in front
 * of flattened stage `stage` (layer * 5 + stage kind; QKV, ATT, WO, GU, DOWN)
 * of later cooperative decode calls waits for one arrival more than the grid
 * makes, so every CTA's bounded wait gives up (after the wait limit) and the
 * call reports DDL_ERR_TIMEOUT through ddl_read_device_status.  No fault, trap
 * or unbounded wait is involved.  -1 turns it off (the default); stage 0 has
 * no barrier in front of it. */
int ddl_test_hold_barrier(int32_t stage);

/* Tracing: when device_buf (device memory) is not NULL, every later decode
 * call of at most 96 layers whose trace fits in `bytes` writes 32 uint64
 * words per (stage, CTA), stages in order (layer * 5 + stage: QKV, ATT, WO,
 * GU, DOWN): word 0 = %globaltimer (ns) at the stage start; words 1..14 =
 * %clock64 (SM cycles) at the end of the stage prologue (word 1), the end
 * of each of the 8 consumer warps' streams (words 2..9), the stage end (word
 * 10), and inside a weight stage's prologue: x copies issued (word 11), x
 * landed (word 13), fragments and RMSNorm factor done (word 14), the
 * prologue's entry (word 12); word 15 = %clock64 at the stage start; words 16..23 = the
 * cycles each consumer warp waited for its ring's data, words 24..31 = the
 * ring slots it consumed.  Needs L * 5 * SMs * 32 * 8 bytes.  NULL turns
 * tracing off. */
int ddl_set_trace(void* device_buf, size_t bytes);

/* Synchronize `stream` and read the device status word of the last decode
 * call that used `workspace` (DDL_OK or DDL_ERR_TIMEOUT); host-blocking.
 * workspace NULL reads the status word of the last ddl_stack_decode_noalloc
 * call (its static scratch).  shape, B and s_max are those of that call. */
int ddl_read_device_status(const void* workspace, const ddl_shape* shape, int32_t B,
                           int64_t s_max, int32_t* status_out, void* stream);

const char* ddl_status_string(int status);

/* The last CUDA error string seen by the library in this process ("" if none). */
const char* ddl_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* DDL_H */
