// Small kernels of the decode step and of context set-up: the embedding
// gather, the RoPE angle table, and the one-time weight repacks.
#include <math.h>

#include "k2_kernels.h"
#include "k2_common.cuh"

namespace k2 {

namespace {

// x = E[token] widened to fp32 (k2-burn README, "Project layout", model.rs:
// embed -> layers).  A token outside [0, vocab) raises GUARD_TOKEN and yields
// a zero row instead of an out-of-bounds read.
template <typename WT>
__global__ void embed_kernel(const WT* __restrict__ E, int vocab, int hidden, const int* __restrict__ tokens,
                             float* __restrict__ resid, unsigned* guard, int* hist, int hist_stride,
                             const int* pos) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int tok = tokens[b];
  if (hist && threadIdx.x == 0) hist[static_cast<size_t>(b) * hist_stride + pos[b]] = tok;
  float* dst = resid + static_cast<size_t>(b) * hidden;
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) atomicOr(guard, GUARD_TOKEN);
    for (int i = threadIdx.x; i < hidden; i += blockDim.x) dst[i] = 0.f;
    return;
  }
  const WT* src = E + static_cast<size_t>(tok) * hidden;
  for (int i = threadIdx.x; i < hidden; i += blockDim.x) dst[i] = to_f32(src[i]);
}

// (cos, sin) of pos * theta^(-2i/d) for every position and pair index
// (k2-burn README, "Status: v0": RoPE "default" type), angles in double.
__global__ void rope_table_kernel(float2* tab, int cap, int half, int d, double theta) {
  const size_t n = static_cast<size_t>(cap) * half;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(idx / half);
    const int i = static_cast<int>(idx % half);
    const double inv = pow(theta, -2.0 * i / d);
    double s, c;
    sincos(static_cast<double>(pos) * inv, &s, &c);
    tab[idx] = make_float2(static_cast<float>(c), static_cast<float>(s));
  }
}

// Fused QKV weight [(nq + 2 nkv) d, hidden] with the rows of every head
// reordered as (0, d/2), (1, d/2 + 1), ...: row 2i of a head is its row i and
// row 2i + 1 its row i + d/2, so the split-half RoPE pairs are adjacent rows.
template <typename WT>
__global__ void repack_qkv_kernel(WT* __restrict__ dst, const WT* __restrict__ wq, const WT* __restrict__ wk,
                                  const WT* __restrict__ wv, int nq, int nkv, int d, int hidden) {
  const int row = blockIdx.x;  // destination row
  const int head = row / d, r = row % d;
  const int src_r = (r & 1) ? (r >> 1) + d / 2 : (r >> 1);
  const WT* src;
  if (head < nq) src = wq + (static_cast<size_t>(head) * d + src_r) * hidden;
  else if (head < nq + nkv) src = wk + (static_cast<size_t>(head - nq) * d + src_r) * hidden;
  else src = wv + (static_cast<size_t>(head - nq - nkv) * d + src_r) * hidden;
  WT* o = dst + static_cast<size_t>(row) * hidden;
  for (int i = threadIdx.x; i < hidden; i += blockDim.x) o[i] = src[i];
}

// gate/up interleaved: row 2i = gate row i, row 2i + 1 = up row i
template <typename WT>
__global__ void repack_gateup_kernel(WT* __restrict__ dst, const WT* __restrict__ wg, const WT* __restrict__ wu,
                                     int hidden) {
  const int row = blockIdx.x;
  const WT* src = ((row & 1) ? wu : wg) + static_cast<size_t>(row >> 1) * hidden;
  WT* o = dst + static_cast<size_t>(row) * hidden;
  for (int i = threadIdx.x; i < hidden; i += blockDim.x) o[i] = src[i];
}

__global__ void advance_kernel(int* seq_len, int seq0, int batch) {
  pdl_wait();
  pdl_trigger();
  const int b = threadIdx.x;
  if (b < batch) seq_len[seq0 + b] += 1;
}

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, cudaStream_t s, bool pdl, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

}  // namespace

cudaError_t launch_embed(const void* E, int wbytes, int vocab, int hidden, const int* tokens, int batch,
                         float* resid, unsigned* guard, int* hist, int hist_stride, const int* pos, cudaStream_t s,
                         bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(batch), dim3(256), s, pdl, attr);
  if (wbytes == 2)
    return cudaLaunchKernelEx(&cfg, embed_kernel<__nv_bfloat16>, static_cast<const __nv_bfloat16*>(E), vocab, hidden,
                              tokens, resid, guard, hist, hist_stride, pos);
  return cudaLaunchKernelEx(&cfg, embed_kernel<float>, static_cast<const float*>(E), vocab, hidden, tokens, resid,
                            guard, hist, hist_stride, pos);
}

cudaError_t launch_rope_table(float2* tab, int cap, int head_dim, double theta, cudaStream_t s) {
  const size_t n = static_cast<size_t>(cap) * (head_dim / 2);
  int blocks = static_cast<int>((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  rope_table_kernel<<<blocks, 256, 0, s>>>(tab, cap, head_dim / 2, head_dim, theta);
  return cudaGetLastError();
}

cudaError_t launch_repack_qkv(void* dst, const void* wq, const void* wk, const void* wv, int wbytes, int nq, int nkv,
                              int d, int hidden, cudaStream_t s) {
  const int rows = (nq + 2 * nkv) * d;
  if (wbytes == 2)
    repack_qkv_kernel<__nv_bfloat16><<<rows, 256, 0, s>>>(
        static_cast<__nv_bfloat16*>(dst), static_cast<const __nv_bfloat16*>(wq), static_cast<const __nv_bfloat16*>(wk),
        static_cast<const __nv_bfloat16*>(wv), nq, nkv, d, hidden);
  else
    repack_qkv_kernel<float><<<rows, 256, 0, s>>>(static_cast<float*>(dst), static_cast<const float*>(wq),
                                                  static_cast<const float*>(wk), static_cast<const float*>(wv), nq,
                                                  nkv, d, hidden);
  return cudaGetLastError();
}

cudaError_t launch_repack_gateup(void* dst, const void* wg, const void* wu, int wbytes, int inter, int hidden,
                                 cudaStream_t s) {
  if (wbytes == 2)
    repack_gateup_kernel<__nv_bfloat16><<<2 * inter, 256, 0, s>>>(
        static_cast<__nv_bfloat16*>(dst), static_cast<const __nv_bfloat16*>(wg), static_cast<const __nv_bfloat16*>(wu),
        hidden);
  else
    repack_gateup_kernel<float><<<2 * inter, 256, 0, s>>>(static_cast<float*>(dst), static_cast<const float*>(wg),
                                                          static_cast<const float*>(wu), hidden);
  return cudaGetLastError();
}

cudaError_t misc_init_attrs() {
  cudaError_t e = set_kernel_smem(embed_kernel<__nv_bfloat16>, 0);
  if (e == cudaSuccess) e = set_kernel_smem(embed_kernel<float>, 0);
  if (e == cudaSuccess) e = set_kernel_smem(advance_kernel, 0);
  return e;
}

cudaError_t launch_advance(int* seq_len, int seq0, int batch, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(1), dim3(32 * ((batch + 31) / 32)), s, pdl, attr);
  return cudaLaunchKernelEx(&cfg, advance_kernel, seq_len, seq0, batch);
}

}  // namespace k2
