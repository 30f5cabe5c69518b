// Prefill of a block of prompt tokens (k2-burn README, "Status: v0": prefill
// then single-token decode; only the last position's logits are needed).
//
// The projections run as tensor-core GEMMs (k2_tcgemm.cu) over the whole
// block; the kernels here do the row-wise work between them:
//   embed rows -> [GroupedRMSNorm -> QKV GEMM -> split-half RoPE + KV append ->
//   causal GQA attention -> o_proj GEMM (+residual) -> GroupedRMSNorm ->
//   gate/up GEMM (+SwiGLU) -> down GEMM (+residual)] x layers.
// Inputs of a GEMM are written as bf16 (hi, lo) pairs whose sum is the fp32
// value (see k2_tcgemm.cu); the residual stream stays fp32.
#include <math.h>

#include <type_traits>

#include <algorithm>
#include <utility>

#include "k2_kernels.h"
#include "k2_common.cuh"

namespace k2 {

namespace {

__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

template <typename WT>
__global__ void embed_rows_kernel(const int* __restrict__ tokens, const WT* __restrict__ E, float* __restrict__ X,
                                  int H, int vocab, unsigned* guard, int* hist, int hist_stride, const int* pos,
                                  int pos0, const int* pos0_dev) {
  const int t = blockIdx.x;
  pdl_wait();  // tokens and lengths come from the previous kernel
  pdl_trigger();
  int tok = tokens[t];
  if (hist && threadIdx.x == 0)
    hist[pos ? static_cast<size_t>(t) * hist_stride + pos[t]
             : static_cast<size_t>(pos0_dev ? *pos0_dev : pos0) + t] = tok;
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) atomicOr(guard, GUARD_TOKEN);
    tok = 0;
  }
  const WT* e = E + static_cast<size_t>(tok) * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x) X[static_cast<size_t>(t) * H + i] = to_f32(e[i]);
}

// GroupedRMSNorm of one row per CTA (k2-burn README, "Model shape": layernorm
// groups), written as bf16 hi/lo, or (f16) as single fp16 into oh.  H is a
// multiple of 4 (every caller's activations are tensor-map rows: a multiple of
// 8); the launch gives each thread one float4 of the row where H <= 4096.
template <typename WT>
__device__ __forceinline__ float4 load4_gain(const WT* g, int i);
template <>
__device__ __forceinline__ float4 load4_gain<__nv_bfloat16>(const __nv_bfloat16* g, int i) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(g + i));
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                     __uint_as_float(v.y & 0xFFFF0000u));
}
template <>
__device__ __forceinline__ float4 load4_gain<float>(const float* g, int i) {
  return __ldg(reinterpret_cast<const float4*>(g + i));
}

template <typename WT>
__global__ void __launch_bounds__(1024)
    norm_rows_kernel(const float* __restrict__ X, const WT* __restrict__ gain, __nv_bfloat16* __restrict__ oh,
                     __nv_bfloat16* __restrict__ ol, int H, int groups, float eps, int rows,
                     float4* __restrict__ zero, size_t zero_n4, float* __restrict__ copy, int f16,
                     unsigned* __restrict__ guard) {
  __shared__ float part[32][4];
  __shared__ float rs[4];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();  // X comes from the previous kernel
  pdl_trigger();
  if (t >= rows) {  // the CTAs past the rows clear the next GEMM's output (zero_n4 float4s)
    for (size_t i = static_cast<size_t>(t - rows) * blockDim.x + tid; i < zero_n4;
         i += static_cast<size_t>(gridDim.x - rows) * blockDim.x)
      zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const float* x = X + static_cast<size_t>(t) * H;
  const int gsz = H / groups;
  float ss[4] = {0.f, 0.f, 0.f, 0.f};
  for (int i = tid * 4; i < H; i += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(x + i);
    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int g = (i + j) / gsz;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q == g) ss[q] += e[j] * e[j];
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) ss[q] = warp_sum(ss[q]);
  if (lane == 0)
    for (int q = 0; q < 4; ++q) part[warp][q] = ss[q];
  __syncthreads();
  if (tid < groups) {
    float sum = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x / 32); ++w) sum += part[w][tid];
    rs[tid] = 1.0f / sqrtf(sum / static_cast<float>(gsz) + eps);
  }
  __syncthreads();
  bool range = false;
  for (int i = tid * 4; i < H; i += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(x + i);  // the same thread's load above: an L1 hit
    const float4 gn = load4_gain<WT>(gain, i);
    const float e[4] = {v.x, v.y, v.z, v.w}, gg[4] = {gn.x, gn.y, gn.z, gn.w};
    float y[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) y[j] = e[j] * rs[(i + j) / gsz] * gg[j];
    const size_t o = static_cast<size_t>(t) * H + i;
    if (f16) {
#pragma unroll
      for (int j = 0; j < 4; ++j) range |= !(fabsf(y[j]) <= 65504.f);
      const __half2 a = __floats2half2_rn(y[0], y[1]), b = __floats2half2_rn(y[2], y[3]);
      uint2 w;
      w.x = *reinterpret_cast<const uint32_t*>(&a);
      w.y = *reinterpret_cast<const uint32_t*>(&b);
      *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(oh) + o) = w;
    } else {
      __nv_bfloat16 hi[4], lo[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) split_bf16(y[j], hi[j], lo[j]);
      *reinterpret_cast<__nv_bfloat162*>(oh + o) = __nv_bfloat162(hi[0], hi[1]);
      *reinterpret_cast<__nv_bfloat162*>(oh + o + 2) = __nv_bfloat162(hi[2], hi[3]);
      *reinterpret_cast<__nv_bfloat162*>(ol + o) = __nv_bfloat162(lo[0], lo[1]);
      *reinterpret_cast<__nv_bfloat162*>(ol + o + 2) = __nv_bfloat162(lo[2], lo[3]);
    }
    if (copy) *reinterpret_cast<float4*>(copy + o) = v;
  }
  if (range && guard != nullptr) atomicOr(guard, GUARD_RANGE);
}

// bf16 -> fp16, eight values per thread and step
__global__ void bf16_to_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n8,
                                   unsigned* __restrict__ guard) {
  bool range = false;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(src + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // a bf16 is the high half of the fp32 with the same value
      float a = __uint_as_float(w[j] << 16), b = __uint_as_float(w[j] & 0xFFFF0000u);
      range |= !(fabsf(a) <= 65504.f) || !(fabsf(b) <= 65504.f);
      a = fminf(fmaxf(a, -65504.f), 65504.f);
      b = fminf(fmaxf(b, -65504.f), 65504.f);
      const __half2 h = __floats2half2_rn(a, b);
      o[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (range) atomicOr(guard, GUARD_RANGE);
}

// split-half RoPE on the QKV GEMM output (rows of every head in the packed
// order (i, i + d/2) adjacent) and the KV append of every token of the block
template <typename KVT>
__global__ void rope_append_kernel(const float* __restrict__ qkv, float* __restrict__ Q, const float2* __restrict__ rope,
                                   KVT* __restrict__ kc, KVT* __restrict__ vc, __half* __restrict__ ks,
                                   __half* __restrict__ vs, int nq, int nkv, int D, int pos0, const int* pos0_dev,
                                   size_t head_row0, int cap) {
  extern __shared__ float rows[];  // [2 * nkv][D]: this token's K and V rows
  pdl_wait();  // qkv comes from the previous kernel
  pdl_trigger();
  const int t = blockIdx.x, tid = threadIdx.x;
  const int qkv_n = (nq + 2 * nkv) * D, half = D / 2, pos = (pos0_dev ? *pos0_dev : pos0) + t;
  const float* src = qkv + static_cast<size_t>(t) * qkv_n;
  for (int idx = tid; idx < (nq + 2 * nkv) * half; idx += blockDim.x) {
    const int h = idx / half, i = idx - h * half;
    float a = src[h * D + 2 * i], b = src[h * D + 2 * i + 1];
    if (h < nq + nkv) {
      const float2 cs = rope[static_cast<size_t>(pos) * half + i];
      const float ra = a * cs.x - b * cs.y, rb = b * cs.x + a * cs.y;
      a = ra;
      b = rb;
    }
    if (h < nq) {
      Q[static_cast<size_t>(t) * nq * D + h * D + i] = a;
      Q[static_cast<size_t>(t) * nq * D + h * D + i + half] = b;
    } else {
      const int r = h - nq;  // K rows 0 .. nkv-1, then V rows
      rows[r * D + i] = a;
      rows[r * D + i + half] = b;
    }
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int r = warp; r < 2 * nkv; r += blockDim.x / 32) {  // one warp per K or V row
    const int g = r < nkv ? r : r - nkv;
    const size_t row = (head_row0 + static_cast<size_t>(g) * cap + pos);
    KVT* dst = (r < nkv ? kc : vc) + row * D;
    const float* v = rows + r * D;
    if constexpr (std::is_same<KVT, int8_t>::value) {
      float amax = 0.f;
      for (int e = lane; e < D; e += 32) amax = fmaxf(amax, fabsf(v[e]));
      amax = warp_max(amax);
      const __half s16 = __float2half_rn(fminf(amax / 127.0f, 65504.0f));
      const float sf = __half2float(s16);
      for (int e = lane; e < D; e += 32) {
        float cq = sf > 0.f ? rintf(v[e] / sf) : 0.f;
        cq = fminf(fmaxf(cq, -127.f), 127.f);
        dst[e] = static_cast<int8_t>(cq);
      }
      if (lane == 0) (r < nkv ? ks : vs)[row] = s16;
    } else if constexpr (std::is_same<KVT, __half>::value) {
      for (int e = lane; e < D; e += 32) dst[e] = __float2half_rn(v[e]);
    } else {
      for (int e = lane; e < D; e += 32) dst[e] = v[e];
    }
  }
}

// Causal GQA attention of a block of query tokens against the cache (which
// already holds the block's own rows).  One CTA per (16 query tokens, KV head):
// the 16 x REP query rows share every 64-key K/V tile; fp32 scores, online
// softmax per row, output written as bf16 hi/lo for the o_proj GEMM.
constexpr int kPaQT = 16, kPaKT = 64, kPaThreads = 256;

template <int D, int REP, typename KVT>
__global__ void __launch_bounds__(kPaThreads) prefill_attn_kernel(const float* __restrict__ Q, const KVT* __restrict__ kc,
                                                                  const KVT* __restrict__ vc, const __half* __restrict__ ks,
                                                                  const __half* __restrict__ vs, __nv_bfloat16* __restrict__ oh,
                                                                  __nv_bfloat16* __restrict__ ol, int n, int nq, int pos0,
                                                                  size_t head_row0, int cap, float scale) {
  constexpr int QR = kPaQT * REP;   // query rows of the CTA (64 for REP 4)
  constexpr int DP = D + 1;         // padded row (bank spread)
  constexpr int RPT = QR / 16;      // rows per thread (threads as 16 x 16)
  constexpr int KPT = kPaKT / 16;   // keys per thread in the score tile
  constexpr int DPT = D / 16;       // output dims per thread
  extern __shared__ float sm[];
  float* Qs = sm;                    // [QR][DP]
  float* Ks = Qs + QR * DP;          // [KT][DP]
  float* Vs = Ks + kPaKT * DP;       // [KT][D]
  float* Ps = Vs + kPaKT * D;        // [QR][KT + 1]
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int t0 = blockIdx.x * kPaQT, g = blockIdx.y;
  const int nt = min(kPaQT, n - t0);
  const size_t hr = head_row0 + static_cast<size_t>(g) * cap;
  // query rows: r = tq * REP + h  ->  token t0 + tq, head g * REP + h
  for (int idx = tid; idx < QR * D; idx += kPaThreads) {
    const int r = idx / D, d = idx - r * D, tq = r / REP, h = r - tq * REP;
    Qs[r * DP + d] = tq < nt ? Q[static_cast<size_t>(t0 + tq) * nq * D + (g * REP + h) * D + d] * scale : 0.f;
  }
  float m[RPT], l[RPT], o[RPT][DPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int j = 0; j < DPT; ++j) o[i][j] = 0.f;
  }
  const int kend = pos0 + t0 + nt;  // keys [0, kend) can be visible to some row of the CTA
  for (int k0 = 0; k0 < kend; k0 += kPaKT) {
    __syncthreads();  // the previous tile is consumed
    for (int idx = tid; idx < kPaKT * D; idx += kPaThreads) {
      const int j = idx / D, d = idx - j * D, key = k0 + j;
      float kv = 0.f, vv = 0.f;
      if (key < kend) {
        kv = to_f32(kc[(hr + key) * D + d]);
        vv = to_f32(vc[(hr + key) * D + d]);
        if constexpr (std::is_same<KVT, int8_t>::value) {
          kv *= __half2float(ks[hr + key]);
          vv *= __half2float(vs[hr + key]);
        }
      }
      Ks[j * DP + d] = kv;
      Vs[j * D + d] = vv;
    }
    __syncthreads();
    // scores of rows ty * RPT + i, keys tx + 16 * c
    float s[RPT][KPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
      for (int c = 0; c < KPT; ++c) s[i][c] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; ++d) {
      float qv[RPT], kv[KPT];
#pragma unroll
      for (int i = 0; i < RPT; ++i) qv[i] = Qs[(ty * RPT + i) * DP + d];
#pragma unroll
      for (int c = 0; c < KPT; ++c) kv[c] = Ks[(tx + 16 * c) * DP + d];
#pragma unroll
      for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int c = 0; c < KPT; ++c) s[i][c] = fmaf(qv[i], kv[c], s[i][c]);
    }
    // causal mask, online softmax (the 16 threads of a row group share a row)
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = ty * RPT + i, tq = r / REP;
      const int qpos = pos0 + t0 + tq;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < KPT; ++c) {
        const int key = k0 + tx + 16 * c;
        if (key > qpos || tq >= nt) s[i][c] = -INFINITY;
        mx = fmaxf(mx, s[i][c]);
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[i], mx);
      const float al = mn == -INFINITY ? 1.f : expf(m[i] - mn);
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < KPT; ++c) {
        const float p = s[i][c] == -INFINITY ? 0.f : expf(s[i][c] - mn);
        Ps[r * (kPaKT + 1) + tx + 16 * c] = p;
        sum += p;
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l[i] = l[i] * al + sum;
      m[i] = mn;
#pragma unroll
      for (int j = 0; j < DPT; ++j) o[i][j] *= al;
    }
    __syncthreads();
    // o[rows][dims tx * DPT ..] += P . V
#pragma unroll 4
    for (int j = 0; j < kPaKT; ++j) {
      float vv[DPT];
#pragma unroll
      for (int e = 0; e < DPT; ++e) vv[e] = Vs[j * D + tx * DPT + e];
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float p = Ps[(ty * RPT + i) * (kPaKT + 1) + j];
#pragma unroll
        for (int e = 0; e < DPT; ++e) o[i][e] = fmaf(p, vv[e], o[i][e]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = ty * RPT + i, tq = r / REP, h = r - tq * REP;
    if (tq >= nt) continue;
    const float inv = 1.0f / l[i];
    const size_t base = static_cast<size_t>(t0 + tq) * nq * D + (g * REP + h) * D + tx * DPT;
#pragma unroll
    for (int e = 0; e < DPT; ++e) {
      __nv_bfloat16 hi, lo;
      split_bf16(o[i][e] * inv, hi, lo);
      oh[base + e] = hi;
      ol[base + e] = lo;
    }
  }
}

// The same causal attention on the tensor cores (mma.sync m16n8k16, fp16 in,
// fp32 accumulate) for fp16 and int8 caches: a CTA of 4 warps takes 64 query
// rows (64 / REP tokens x REP heads of one KV head), each warp 16 rows.  K/V
// tiles of 64 keys sit in shared memory as fp16 (int8 codes are exact in fp16;
// their scales multiply the scores' and probabilities' columns), with 16-byte
// chunks XOR-swizzled by row so that ldmatrix reads are conflict-free.  The
// query rows and the probabilities enter each MMA as two fp16 halves (hi + lo),
// which keeps ~22 mantissa bits: the result matches fp32 CUDA-core arithmetic
// to ~1e-6.  The score accumulators are reused as the probability fragments
// of the P.V product (same register layout).
constexpr int kMaRows = 64, kMaKT = 64, kMaThreads = 128;

// byte offset of 16-byte chunk `c` of row `r` in a swizzled [rows][D] fp16 tile
template <int D>
__device__ __forceinline__ int swz(int r, int c) {
  return r * (D * 2) + ((c ^ (r & 7)) << 4);
}

template <int D, int REP, typename KVT>
__global__ void __launch_bounds__(kMaThreads) prefill_attn_mma_kernel(
    const float* __restrict__ Q, const KVT* __restrict__ kc, const KVT* __restrict__ vc, const __half* __restrict__ ks,
    const __half* __restrict__ vs, __nv_bfloat16* __restrict__ oh, __nv_bfloat16* __restrict__ ol, int n, int nq,
    int pos0, size_t head_row0, int cap, float scale) {
  constexpr bool I8 = std::is_same<KVT, int8_t>::value;
  constexpr int QT = kMaRows / REP;  // tokens per CTA
  constexpr int KS = D / 16;         // k-steps of Q.K
  constexpr int NT = D / 8;          // n-tiles of P.V
  constexpr int CH = D / 8;          // 16-byte chunks per fp16 row
  __shared__ __align__(128) __half Ks[kMaKT * D];
  __shared__ __align__(128) __half Vs[kMaKT * D];
  __shared__ float ksc[kMaKT], vsc[kMaKT];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int t0 = blockIdx.x * QT, kvh = blockIdx.y;
  const int nt = min(QT, n - t0);
  const size_t hr = head_row0 + static_cast<size_t>(kvh) * cap;
  // this thread's two query rows (r and r + 8 of the warp's 16)
  const int r0 = warp * 16 + g, r1 = r0 + 8;
  const int tq0 = r0 / REP, tq1 = r1 / REP;
  const int qpos0 = pos0 + t0 + tq0, qpos1 = pos0 + t0 + tq1;
  // query fragments (hi, lo): rows r0/r1, dims 16 kk + 2t (+1), + 8
  uint32_t qh[KS][4], qlo[KS][4];
  {
    auto qv = [&](int r, int d) -> float {
      const int tq = r / REP, h = r - tq * REP;
      return tq < nt ? Q[static_cast<size_t>(t0 + tq) * nq * D + (kvh * REP + h) * D + d] * scale : 0.f;
    };
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int d0 = 16 * kk + 2 * t;
      split_half2(qv(r0, d0), qv(r0, d0 + 1), qh[kk][0], qlo[kk][0]);
      split_half2(qv(r1, d0), qv(r1, d0 + 1), qh[kk][1], qlo[kk][1]);
      split_half2(qv(r0, d0 + 8), qv(r0, d0 + 9), qh[kk][2], qlo[kk][2]);
      split_half2(qv(r1, d0 + 8), qv(r1, d0 + 9), qh[kk][3], qlo[kk][3]);
    }
  }
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const uint32_t ks_base = smem_u32(Ks), vs_base = smem_u32(Vs);
  const int kend = pos0 + t0 + nt;
  for (int k0 = 0; k0 < kend; k0 += kMaKT) {
    __syncthreads();  // the previous tile is consumed
    for (int idx = tid; idx < kMaKT * CH; idx += kMaThreads) {
      const int r = idx / CH, c = idx - r * CH, key = k0 + r;
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (key < kend) {
        if constexpr (I8) {  // 8 codes -> 8 halves
          const uint2 kq = *reinterpret_cast<const uint2*>(kc + (hr + key) * D + c * 8);
          const uint2 vq = *reinterpret_cast<const uint2*>(vc + (hr + key) * D + c * 8);
          auto cvt = [](uint2 q) {
            uint32_t w[4];
            const uint32_t x[2] = {q.x, q.y};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float a = static_cast<float>(static_cast<int8_t>((x[i >> 1] >> (16 * (i & 1))) & 0xFF));
              const float b = static_cast<float>(static_cast<int8_t>((x[i >> 1] >> (16 * (i & 1) + 8)) & 0xFF));
              w[i] = pack_half2(a, b);
            }
            return make_uint4(w[0], w[1], w[2], w[3]);
          };
          kv = cvt(kq);
          vv = cvt(vq);
        } else {
          kv = *reinterpret_cast<const uint4*>(kc + (hr + key) * D + c * 8);
          vv = *reinterpret_cast<const uint4*>(vc + (hr + key) * D + c * 8);
        }
      }
      *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(Ks) + swz<D>(r, c)) = kv;
      *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(Vs) + swz<D>(r, c)) = vv;
    }
    if (tid < kMaKT) {
      const int key = k0 + tid;
      ksc[tid] = I8 && key < kend ? __half2float(ks[hr + key]) : 1.f;
      vsc[tid] = I8 && key < kend ? __half2float(vs[hr + key]) : 1.f;
    }
    __syncthreads();
    // S = Q K^T over the 64 keys: 8 n-tiles of 8 keys
    float sc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const int m = lane >> 3, rr = lane & 7;
        const int key = 8 * (j + (m >> 1)) + rr, chunk = 2 * kk + (m & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ks_base + swz<D>(key, chunk), b0, b1, b2, b3);
        mma16816(sc[j], qh[kk], b0, b1);
        mma16816(sc[j], qlo[kk], b0, b1);
        mma16816(sc[j + 1], qh[kk], b2, b3);
        mma16816(sc[j + 1], qlo[kk], b2, b3);
      }
    }
    // scales (int8), causal mask, online softmax of rows r0 (c0, c1) and r1 (c2, c3)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kl = 8 * j + 2 * t + e, key = k0 + kl;
        const float ksf = I8 ? ksc[kl] : 1.f;
        sc[j][e] = (key > qpos0 || tq0 >= nt) ? -INFINITY : sc[j][e] * ksf;
        sc[j][2 + e] = (key > qpos1 || tq1 >= nt) ? -INFINITY : sc[j][2 + e] * ksf;
        mx0 = fmaxf(mx0, sc[j][e]);
        mx1 = fmaxf(mx1, sc[j][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = mn0 == -INFINITY ? 1.f : expf(m0 - mn0), al1 = mn1 == -INFINITY ? 1.f : expf(m1 - mn1);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[j][e] = sc[j][e] == -INFINITY ? 0.f : expf(sc[j][e] - mn0);
        sc[j][2 + e] = sc[j][2 + e] == -INFINITY ? 0.f : expf(sc[j][2 + e] - mn1);
        s0 += sc[j][e];
        s1 += sc[j][2 + e];
      }
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    l0 = l0 * al0 + s0;
    l1 = l1 * al1 + s1;
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      o[j][0] *= al0;
      o[j][1] *= al0;
      o[j][2] *= al1;
      o[j][3] *= al1;
    }
    // O += P V: k-steps of 16 keys (score n-tiles 2kk, 2kk+1), n-tiles of 8 dims
#pragma unroll
    for (int kk = 0; kk < kMaKT / 16; ++kk) {
      uint32_t ph[4], pl[4];
      {
        const int ka = 16 * kk + 2 * t, kb = ka + 8;
        const float va0 = I8 ? vsc[ka] : 1.f, va1 = I8 ? vsc[ka + 1] : 1.f;
        const float vb0 = I8 ? vsc[kb] : 1.f, vb1 = I8 ? vsc[kb + 1] : 1.f;
        split_half2(sc[2 * kk][0] * va0, sc[2 * kk][1] * va1, ph[0], pl[0]);
        split_half2(sc[2 * kk][2] * va0, sc[2 * kk][3] * va1, ph[1], pl[1]);
        split_half2(sc[2 * kk + 1][0] * vb0, sc[2 * kk + 1][1] * vb1, ph[2], pl[2]);
        split_half2(sc[2 * kk + 1][2] * vb0, sc[2 * kk + 1][3] * vb1, ph[3], pl[3]);
      }
#pragma unroll
      for (int j = 0; j < NT; j += 2) {
        const int m = lane >> 3, rr = lane & 7;
        const int key = 16 * kk + 8 * (m & 1) + rr, chunk = j + (m >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vs_base + swz<D>(key, chunk), b0, b1, b2, b3);
        mma16816(o[j], ph, b0, b1);
        mma16816(o[j], pl, b0, b1);
        mma16816(o[j + 1], ph, b2, b3);
        mma16816(o[j + 1], pl, b2, b3);
      }
    }
  }
  // normalise and write rows r0, r1 (dims 8j + 2t, +1) as bf16 hi/lo
  const float inv0 = l0 > 0.f ? 1.0f / l0 : 0.f, inv1 = l1 > 0.f ? 1.0f / l1 : 0.f;
#pragma unroll
  for (int row = 0; row < 2; ++row) {
    const int r = row ? r1 : r0, tq = r / REP, h = r - tq * REP;
    if (tq >= nt) continue;
    const float inv = row ? inv1 : inv0;
    const size_t base = static_cast<size_t>(t0 + tq) * nq * D + (kvh * REP + h) * D;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        __nv_bfloat16 hi, lo;
        split_bf16(o[j][2 * row + e] * inv, hi, lo);
        oh[base + 8 * j + 2 * t + e] = hi;
        ol[base + 8 * j + 2 * t + e] = lo;
      }
    }
  }
}

template <int D, int REP>
constexpr size_t attn_smem() {
  return sizeof(float) * (static_cast<size_t>(kPaQT * REP) * (D + 1) + kPaKT * (D + 1) + kPaKT * D +
                          kPaQT * REP * (kPaKT + 1));
}

__global__ void advance_by_kernel(int* seq_len, int seq, int n) { seq_len[seq] += n; }

// gate/up GEMM rows (2p, 2p+1) = (gate_p, up_p) -> silu(gate) * up as bf16 hi/lo
__global__ void swiglu_rows_kernel(const float* __restrict__ gu, __nv_bfloat16* __restrict__ oh,
                                   __nv_bfloat16* __restrict__ ol, int I) {
  const float* r = gu + static_cast<size_t>(blockIdx.y) * 2 * I;
  const size_t base = static_cast<size_t>(blockIdx.y) * I;
  pdl_wait();
  pdl_trigger();
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < I; p += gridDim.x * blockDim.x) {
    const float g = r[2 * p], u = r[2 * p + 1];
    __nv_bfloat16 hi, lo;
    split_bf16(g / (1.0f + expf(-g)) * u, hi, lo);
    oh[base + p] = hi;
    ol[base + p] = lo;
  }
}

// fp32 rows -> bf16 (hi, lo) rows
__global__ void rows_hilo_kernel(const float* __restrict__ x, __nv_bfloat16* __restrict__ oh,
                                 __nv_bfloat16* __restrict__ ol, int K) {
  const size_t base = static_cast<size_t>(blockIdx.y) * K;
  pdl_wait();
  pdl_trigger();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < K; i += gridDim.x * blockDim.x) {
    __nv_bfloat16 hi, lo;
    split_bf16(x[base + i], hi, lo);
    oh[base + i] = hi;
    ol[base + i] = lo;
  }
}

// first index of the maximum of each logits row (kimi-k3-in-c k3_run.c,
// `argmax_`), in two passes: kArgChunks partial maxima per row, then one per
// row; a NaN sets the guard and token 0 is written
constexpr int kArgChunks = 64;

__device__ __forceinline__ void best_of(float& v, int& i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) {
    v = ov;
    i = oi;
  }
}

__device__ __forceinline__ void block_best(float& v, int& i, float* sv, int* si) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best_of(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
  if ((threadIdx.x & 31) == 0) {
    sv[threadIdx.x >> 5] = v;
    si[threadIdx.x >> 5] = i;
  }
  __syncthreads();
  if (threadIdx.x == 0)
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) best_of(v, i, sv[w], si[w]);
}

__global__ void argmax_part_kernel(const float* __restrict__ logits, int V, float* __restrict__ pv,
                                   int* __restrict__ pi, int stride, unsigned* guard) {
  __shared__ float sv[32];
  __shared__ int si[32];
  const int row = blockIdx.y, chunk = blockIdx.x;
  const int lo = static_cast<int>((static_cast<long long>(V) * chunk) / gridDim.x);
  const int hi = static_cast<int>((static_cast<long long>(V) * (chunk + 1)) / gridDim.x);
  const float* r = logits + static_cast<size_t>(row) * V;
  pdl_wait();
  pdl_trigger();
  float v = -INFINITY;
  int idx = 0x7fffffff;
  bool nan = false;
  for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    const float x = r[i];
    if (x != x) nan = true;
    else if (x > v) {  // increasing i per thread: its first maximum is kept
      v = x;
      idx = i;
    }
  }
  if (__syncthreads_or(nan) && threadIdx.x == 0) atomicOr(guard, GUARD_NAN);
  block_best(v, idx, sv, si);
  if (threadIdx.x == 0) {
    pv[static_cast<size_t>(row) * stride + chunk] = v;
    pi[static_cast<size_t>(row) * stride + chunk] = idx;
  }
}

__global__ void argmax_final_kernel(const float* __restrict__ pv, const int* __restrict__ pi, int chunks, int stride,
                                    int* __restrict__ next) {
  __shared__ float sv[32];
  __shared__ int si[32];
  pdl_wait();
  pdl_trigger();
  float v = -INFINITY;
  int idx = 0x7fffffff;
  for (int c = threadIdx.x; c < chunks; c += blockDim.x)
    best_of(v, idx, pv[static_cast<size_t>(blockIdx.x) * stride + c], pi[static_cast<size_t>(blockIdx.x) * stride + c]);
  block_best(v, idx, sv, si);
  if (threadIdx.x == 0) next[blockIdx.x] = idx == 0x7fffffff ? 0 : idx;
}


#define K2_PREFILL_ATTN_SHAPES(X) X(128, 4) X(64, 4)

}  // namespace

bool prefill_attn_supported(int head_dim, int rep) {
#define K2_PA_SUP(D, R) \
  if (head_dim == D && rep == R) return true;
  K2_PREFILL_ATTN_SHAPES(K2_PA_SUP)
#undef K2_PA_SUP
  return false;
}

cudaError_t prefill_init_attrs() {
  cudaError_t e = cudaSuccess;
#define K2_PA_ATTR(D, R)                                                                                     \
  if (!e) e = cudaFuncSetAttribute(prefill_attn_kernel<D, R, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                   static_cast<int>(attn_smem<D, R>()));                                    \
  if (!e) e = cudaFuncSetAttribute(prefill_attn_kernel<D, R, __half>,                                        \
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(attn_smem<D, R>())); \
  if (!e) e = cudaFuncSetAttribute(prefill_attn_kernel<D, R, int8_t>,                                        \
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(attn_smem<D, R>()));
  K2_PREFILL_ATTN_SHAPES(K2_PA_ATTR)
#undef K2_PA_ATTR
  if (!e) e = tc_gemm_init_attrs();
  if (!e) e = prefill_attn_tc_init_attrs();
  return e;
}

namespace {
// A launch with programmatic dependent launch when `pdl` (the kernel waits for
// its predecessor with griddepcontrol.wait before reading what it wrote).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
}  // namespace

cudaError_t launch_embed_rows(const int* tokens, int n, const void* E, int wbytes, float* X, int H, int vocab,
                              unsigned* guard, int* hist, int hist_stride, const int* pos, int pos0,
                              const int* pos0_dev, cudaStream_t s, bool pdl) {
  if (wbytes == 2)
    return launch_k(embed_rows_kernel<__nv_bfloat16>, dim3(n), dim3(256), 0, s, pdl, tokens,
                    static_cast<const __nv_bfloat16*>(E), X, H, vocab, guard, hist, hist_stride, pos, pos0, pos0_dev);
  return launch_k(embed_rows_kernel<float>, dim3(n), dim3(256), 0, s, pdl, tokens, static_cast<const float*>(E), X, H,
                  vocab, guard, hist, hist_stride, pos, pos0, pos0_dev);
}

cudaError_t launch_bf16_to_f16(__half* dst, const __nv_bfloat16* src, size_t n, unsigned* guard, cudaStream_t s) {
  if (n % 8 || reinterpret_cast<uintptr_t>(dst) % 16 || reinterpret_cast<uintptr_t>(src) % 16)
    return cudaErrorInvalidValue;
  const size_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<size_t>((n8 + 255) / 256, 152 * 8));
  bf16_to_f16_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), n8,
                                          guard);
  return cudaGetLastError();
}

cudaError_t launch_norm_rows(const float* X, int n, const void* gain, int wbytes, __nv_bfloat16* oh,
                             __nv_bfloat16* ol, int H, int groups, float eps, cudaStream_t s, bool pdl, float* zero,
                             size_t zero_floats, float* copy, bool f16, unsigned* guard) {
  if (zero_floats % 4 || (zero_floats && reinterpret_cast<uintptr_t>(zero) % 16) || H % 4 || groups < 1 || groups > 4)
    return cudaErrorInvalidValue;
  const size_t n4 = zero_floats / 4;
  // extra CTAs (up to one per 8192 float4s, at most 64) clear the next GEMM's output
  const int zc = n4 ? static_cast<int>(std::min<size_t>(64, (n4 + 8191) / 8192)) : 0;
  // one float4 per thread (H <= 4096), in whole warps
  const int threads = std::min(1024, std::max(32, (H / 4 + 31) / 32 * 32));
  if (wbytes == 2)
    return launch_k(norm_rows_kernel<__nv_bfloat16>, dim3(n + zc), dim3(threads), 0, s, pdl, X,
                    static_cast<const __nv_bfloat16*>(gain), oh, ol, H, groups, eps, n,
                    reinterpret_cast<float4*>(zero), n4, copy, f16 ? 1 : 0, guard);
  return launch_k(norm_rows_kernel<float>, dim3(n + zc), dim3(threads), 0, s, pdl, X,
                  static_cast<const float*>(gain), oh,
                  ol, H, groups, eps, n, reinterpret_cast<float4*>(zero), n4, copy, f16 ? 1 : 0, guard);
}

cudaError_t launch_rope_append(const float* qkv, float* Q, const float2* rope, int kv_dtype, void* kc, void* vc,
                               void* ks, void* vs, int n, int nq, int nkv, int D, int pos0, const int* pos0_dev,
                               size_t head_row0, int cap, cudaStream_t s, bool pdl) {
  const size_t smem = sizeof(float) * 2 * nkv * D;
  switch (kv_dtype) {
    case 0:
      return launch_k(rope_append_kernel<float>, dim3(n), dim3(256), smem, s, pdl, qkv, Q, rope, static_cast<float*>(kc),
                      static_cast<float*>(vc), static_cast<__half*>(nullptr), static_cast<__half*>(nullptr), nq, nkv, D,
                      pos0, pos0_dev, head_row0, cap);
    case 2:
      return launch_k(rope_append_kernel<__half>, dim3(n), dim3(256), smem, s, pdl, qkv, Q, rope,
                      static_cast<__half*>(kc), static_cast<__half*>(vc), static_cast<__half*>(nullptr),
                      static_cast<__half*>(nullptr), nq, nkv, D, pos0, pos0_dev, head_row0, cap);
    default:
      return launch_k(rope_append_kernel<int8_t>, dim3(n), dim3(256), smem, s, pdl, qkv, Q, rope,
                      static_cast<int8_t*>(kc), static_cast<int8_t*>(vc), static_cast<__half*>(ks),
                      static_cast<__half*>(vs), nq, nkv, D, pos0, pos0_dev, head_row0, cap);
  }
}

cudaError_t launch_prefill_attn(const float* Q, int kv_dtype, const void* kc, const void* vc, const void* ks,
                                const void* vs, __nv_bfloat16* oh, __nv_bfloat16* ol, int n, int nq, int nkv, int D,
                                int pos0, size_t head_row0, int cap, float scale, cudaStream_t s) {
  const int rep = nq / nkv;
  dim3 grid((n + kPaQT - 1) / kPaQT, nkv);
#define K2_PA_LAUNCH(DD, R)                                                                                       \
  if (D == DD && rep == R) {                                                                                      \
    const size_t sm = attn_smem<DD, R>();                                                                         \
    const dim3 mgrid((n + kMaRows / R - 1) / (kMaRows / R), nkv);                                              \
    if (kv_dtype == 0)                                                                                            \
      prefill_attn_kernel<DD, R, float><<<grid, kPaThreads, sm, s>>>(                                             \
          Q, static_cast<const float*>(kc), static_cast<const float*>(vc), nullptr, nullptr, oh, ol, n, nq, pos0, \
          head_row0, cap, scale);                                                                                 \
    else if (kv_dtype == 2)                                                                                       \
      prefill_attn_mma_kernel<DD, R, __half><<<mgrid, kMaThreads, 0, s>>>(                                        \
          Q, static_cast<const __half*>(kc), static_cast<const __half*>(vc), nullptr, nullptr, oh, ol, n, nq,     \
          pos0, head_row0, cap, scale);                                                                           \
    else                                                                                                          \
      prefill_attn_mma_kernel<DD, R, int8_t><<<mgrid, kMaThreads, 0, s>>>(                                        \
          Q, static_cast<const int8_t*>(kc), static_cast<const int8_t*>(vc), static_cast<const __half*>(ks),      \
          static_cast<const __half*>(vs), oh, ol, n, nq, pos0, head_row0, cap, scale);                            \
    return cudaGetLastError();                                                                                    \
  }
  K2_PREFILL_ATTN_SHAPES(K2_PA_LAUNCH)
#undef K2_PA_LAUNCH
  return cudaErrorInvalidValue;
}

cudaError_t launch_swiglu_rows(const float* gu, __nv_bfloat16* oh, __nv_bfloat16* ol, int rows, int I, cudaStream_t s,
                               bool pdl) {
  return launch_k(swiglu_rows_kernel, dim3((I + 255) / 256, rows), dim3(256), 0, s, pdl, gu, oh, ol, I);
}

cudaError_t launch_rows_hilo(const float* x, __nv_bfloat16* oh, __nv_bfloat16* ol, int rows, int K, cudaStream_t s,
                             bool pdl) {
  return launch_k(rows_hilo_kernel, dim3((K + 255) / 256, rows), dim3(256), 0, s, pdl, x, oh, ol, K);
}

cudaError_t launch_argmax_rows(const float* logits, int rows, int V, int* next, float* part_val, int* part_idx,
                               int part_stride, unsigned* guard, cudaStream_t s, bool pdl) {
  if (part_stride < kArgChunks) return cudaErrorInvalidValue;
  cudaError_t e = launch_k(argmax_part_kernel, dim3(kArgChunks, rows), dim3(256), 0, s, pdl, logits, V, part_val,
                           part_idx, part_stride, guard);
  if (e != cudaSuccess) return e;
  return launch_k(argmax_final_kernel, dim3(rows), dim3(64), 0, s, pdl, static_cast<const float*>(part_val),
                  static_cast<const int*>(part_idx), static_cast<int>(kArgChunks), part_stride, next);
}

cudaError_t launch_advance_by(int* seq_len, int seq, int n, cudaStream_t s) {
  advance_by_kernel<<<1, 1, 0, s>>>(seq_len, seq, n);
  return cudaGetLastError();
}

}  // namespace k2
