// ddl_pack.cu -- weight and cache preparation: the symmetric INT4 quantizer,
// the canonical -> kernel-native packer, and the KV-cache append.
#include <cuda_bf16.h>
#include <stdio.h>

#include "ddl_device.cuh"
#include "ddl_internal.h"

namespace ddl {

// ------------------------------------------------------------------ quantizer
// One warp per (row, group of 64): lane l owns columns 2l, 2l+1.
// s = bf16_rne(absmax / 7) (fp32 division, correctly rounded; absmax/7 of a
// bf16 value is never an fp32 or bf16 tie, so this equals one rounding of the
// exact quotient), code = clamp(rne(w / s), -7, 7), zero group -> s = 0.
__global__ void quantize_int4_kernel(const uint16_t* __restrict__ w, int64_t N, int64_t K,
                                     uint8_t* __restrict__ q, uint16_t* __restrict__ s) {
  const int64_t G = K / DDL_GROUP;
  const int64_t item = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (item >= N * G) return;
  const int lane = threadIdx.x & 31;
  const int64_t n = item / G, g = item % G;
  const uint32_t pair = *reinterpret_cast<const uint32_t*>(w + n * K + g * DDL_GROUP + 2 * lane);
  const float w0 = bf16lo_f32(pair), w1 = bf16hi_f32(pair);
  float amax = fmaxf(fabsf(w0), fabsf(w1));
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, o));
  const uint16_t sb = f32_to_bf16_bits(__fdiv_rn(amax, 7.0f));
  const float sv = bf16_bits_to_f32(sb);
  int c0 = 0, c1 = 0;
  if (sv != 0.f) {
    c0 = (int)fminf(7.f, fmaxf(-7.f, rintf(__fdiv_rn(w0, sv))));
    c1 = (int)fminf(7.f, fmaxf(-7.f, rintf(__fdiv_rn(w1, sv))));
  }
  q[n * (K / 2) + g * (DDL_GROUP / 2) + lane] = (uint8_t)((c0 & 0xF) | ((c1 & 0xF) << 4));
  if (lane == 0) s[n * G + g] = sb;
}

// ------------------------------------------------------------------ packer
struct SrcRows {  // up to three canonical matrices stacked along N
  const uint8_t* q[3];
  const uint16_t* s[3];
  const uint16_t* w[3];
  int32_t rows[3];
};

__device__ __forceinline__ int src_of(const SrcRows& src, int kind, int T, int r, int hd,
                                      int& row) {
  int R = tile_row(kind, T, r, hd);
  if (kind == MK_GU) {
    row = R;
    return r < 8 ? 0 : 1;
  }
  int m = 0;
  while (m < 2 && R >= src.rows[m]) {
    R -= src.rows[m];
    ++m;
  }
  row = R;
  return m;
}

__device__ __forceinline__ uint32_t nib(const SrcRows& src, int m, int row, int K, int k) {
  uint8_t byte = src.q[m][(int64_t)row * (K / 2) + k / 2];
  return (k & 1) ? (byte >> 4) : (byte & 0xF);
}

// One thread per 32-bit word of the code stream, then per scale word.
__global__ void pack_int4_kernel(MatGeom m, int kind, int hd, SrcRows src,
                                 uint32_t* __restrict__ wout, uint32_t* __restrict__ sout) {
  const int64_t nw = m.T * 128, ns = m.T * 8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nw + ns;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < nw) {
      const int64_t b = i / 128;
      const int lane = (int)(i % 128) / 4, j = (int)(i % 4);
      const int g = lane / 4, t = lane % 4;
      int kc, T, gi;
      block_coord(m, b, kc, T, gi);
      const int k0 = (kc * m.Gc + gi) * DDL_GROUP + 16 * j + 2 * t;
      int rg, rh;
      const int mg_ = src_of(src, kind, T, g, hd, rg), mh = src_of(src, kind, T, g + 8, hd, rh);
      uint32_t wd = 0;
      wd |= nib(src, mg_, rg, m.K, k0) << 0;
      wd |= nib(src, mh, rh, m.K, k0) << 4;
      wd |= nib(src, mg_, rg, m.K, k0 + 8) << 8;
      wd |= nib(src, mh, rh, m.K, k0 + 8) << 12;
      wd |= nib(src, mg_, rg, m.K, k0 + 1) << 16;
      wd |= nib(src, mh, rh, m.K, k0 + 1) << 20;
      wd |= nib(src, mg_, rg, m.K, k0 + 9) << 24;
      wd |= nib(src, mh, rh, m.K, k0 + 9) << 28;
      wout[b * (QBLK_BYTES / 4) + lane * 4 + j] = wd;
    } else {
      const int64_t si = i - nw, b = si / 8;
      const int g = (int)(si % 8);
      int kc, T, gi;
      block_coord(m, b, kc, T, gi);
      const int grp = kc * m.Gc + gi;
      int rg, rh;
      const int mg_ = src_of(src, kind, T, g, hd, rg), mh = src_of(src, kind, T, g + 8, hd, rh);
      const uint32_t lo = src.s[mg_][(int64_t)rg * m.G + grp], hi = src.s[mh][(int64_t)rh * m.G + grp];
      sout[b * (QBLK_BYTES / 4) + g] = lo | (hi << 16);
    }
  }
}

// bf16 weights: one thread per 32-bit word (two bf16) of a 2048-byte block:
// 4 sub-blocks j of 16 columns, lane (g, t) holds the m16n8k16 A fragment
// {row g k 2t..2t+1, row g+8 k 2t..2t+1, row g k 2t+8..9, row g+8 k 2t+8..9}.
__global__ void pack_bf16_kernel(MatGeom m, int kind, int hd, SrcRows src,
                                 uint32_t* __restrict__ wout) {
  const int64_t nw = m.T * 512;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nw;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / 512;
    const int j = (int)(i % 512) / 128, lane = (int)(i % 128) / 4, reg = (int)(i % 4);
    const int g = lane / 4, t = lane % 4;
    int kc, T, gi;
    block_coord(m, b, kc, T, gi);
    const int k = (kc * m.Gc + gi) * DDL_GROUP + 16 * j + 2 * t + ((reg & 2) ? 8 : 0);
    int row;
    const int ms = src_of(src, kind, T, (reg & 1) ? g + 8 : g, hd, row);
    wout[i] = *reinterpret_cast<const uint32_t*>(src.w[ms] + (int64_t)row * m.K + k);
  }
}

// ------------------------------------------------------------------ KV append
__global__ void kv_append_kernel(uint16_t* __restrict__ kc, uint16_t* __restrict__ vc,
                                 int64_t s_max, int B, int Hkv, int hd, int64_t pos,
                                 const uint16_t* __restrict__ kn, const uint16_t* __restrict__ vn) {
  const int64_t n = (int64_t)B * Hkv * hd;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bh = i / hd, d = i % hd;
    const int64_t dst = (bh * s_max + pos) * hd + d;
    kc[dst] = kn[i];
    vc[dst] = vn[i];
  }
}

}  // namespace ddl

using namespace ddl;

extern "C" int ddl_quantize_int4(const uint16_t* w_bf16, int64_t N, int64_t K, uint8_t* q_out,
                                 uint16_t* scale_out, void* stream) {
  if (!w_bf16 || !q_out || !scale_out || N <= 0 || K <= 0) return DDL_ERR_ARG;
  if (K % DDL_GROUP) return DDL_ERR_SHAPE;
  if (((uintptr_t)w_bf16 & 3) || ((uintptr_t)scale_out & 1)) return DDL_ERR_ALIGN;
  const int64_t items = N * (K / DDL_GROUP);
  const int64_t blocks = (items + 7) / 8;
  if (blocks > 0x7fffffffLL) return DDL_ERR_SHAPE;
  quantize_int4_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(w_bf16, N, K, q_out,
                                                                           scale_out);
  return cuda_status(cudaGetLastError());
}

extern "C" size_t ddl_packed_layer_bytes(const ddl_shape* shape, ddl_wtype wtype) {
  if (check_shape(shape) != DDL_OK || (wtype != DDL_W_INT4 && wtype != DDL_W_BF16)) return 0;
  MatGeom mg[4];
  return (size_t)make_geoms(*shape, wtype, mg);
}

extern "C" int ddl_pack_layer(const ddl_shape* shape, ddl_wtype wtype, const ddl_layer_src* src,
                              void* packed_out, void* stream) {
  int st = check_shape(shape);
  if (st) return st;
  if (!src || !packed_out) return DDL_ERR_ARG;
  if (wtype != DDL_W_INT4 && wtype != DDL_W_BF16) return DDL_ERR_UNSUPPORTED;
  if (!aligned16(packed_out)) return DDL_ERR_ALIGN;
  MatGeom mg[4];
  make_geoms(*shape, wtype, mg);
  const ddl_mat* mats[4][3] = {{&src->wq, &src->wk, &src->wv},
                               {&src->wo, nullptr, nullptr},
                               {&src->wg, &src->wu, nullptr},
                               {&src->wd, nullptr, nullptr}};
  const int32_t Nq = shape->H_q * shape->head_dim, Nkv = shape->H_kv * shape->head_dim;
  const int32_t rows[4][3] = {{Nq, Nkv, Nkv}, {shape->D, 0, 0}, {shape->d_ff, shape->d_ff, 0},
                              {shape->D, 0, 0}};
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* base = (uint8_t*)packed_out;
  for (int k = 0; k < 4; ++k) {
    SrcRows sr;
    memset(&sr, 0, sizeof sr);
    for (int i = 0; i < 3; ++i) {
      if (!mats[k][i]) continue;
      sr.q[i] = mats[k][i]->q;
      sr.s[i] = mats[k][i]->scale;
      sr.w[i] = mats[k][i]->w;
      sr.rows[i] = rows[k][i];
      if (wtype == DDL_W_INT4 && (!sr.q[i] || !sr.s[i])) return DDL_ERR_ARG;
      if (wtype == DDL_W_BF16 && !sr.w[i]) return DDL_ERR_ARG;
      if (wtype == DDL_W_BF16 && ((uintptr_t)sr.w[i] & 3)) return DDL_ERR_ALIGN;
    }
    const int64_t work = mg[k].T * (wtype == DDL_W_INT4 ? 136 : 512);
    const int blocks = (int)((work + 255) / 256 < 65535 * 16 ? (work + 255) / 256 : 65535 * 16);
    if (wtype == DDL_W_INT4)
      pack_int4_kernel<<<blocks, 256, 0, s>>>(mg[k], k, shape->head_dim, sr,
                                              (uint32_t*)(base + mg[k].woff),
                                              (uint32_t*)(base + mg[k].soff));
    else
      pack_bf16_kernel<<<blocks, 256, 0, s>>>(mg[k], k, shape->head_dim, sr,
                                              (uint32_t*)(base + mg[k].woff));
    st = cuda_status(cudaGetLastError());
    if (st) return st;
  }
  return DDL_OK;
}

extern "C" int ddl_kv_append(const ddl_kv* kv, int32_t B, int32_t H_kv, int32_t head_dim,
                             int64_t pos, const uint16_t* k_new, const uint16_t* v_new,
                             void* stream) {
  if (!kv || !kv->k || !kv->v || !k_new || !v_new || B <= 0 || H_kv <= 0 || head_dim <= 0)
    return DDL_ERR_ARG;
  if (pos < 0 || pos >= kv->s_max) return DDL_ERR_POS;
  const int64_t n = (int64_t)B * H_kv * head_dim;
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  kv_append_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(kv->k, kv->v, kv->s_max, B, H_kv,
                                                             head_dim, pos, k_new, v_new);
  return cuda_status(cudaGetLastError());
}
