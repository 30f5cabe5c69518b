// Split-K flash-decode GQA attention for one new token per sequence, with the
// KV-cache append of that token fused in.
//
// What it computes (k2-burn README, "Status: v0" GQA attention, "Limitations"
// plain SDPA with an fp32 softmax, "Model shape" 32 q heads over 8 KV heads):
// for query head h of the new token at position pos, with KV head
// g = h / REP, o_h = softmax_j(q_h . k_j / sqrt(D)) . v_j over j = 0..pos.
//
// Layout and schedule:
//   * grid = (splits, KV heads, sequences); a CTA owns one KV head of one
//     sequence and a contiguous key range, so every K/V byte is read from HBM
//     once per step and shared by the REP query heads of its group;
//   * the key range is streamed in 64-key tiles through a ring of shared-memory
//     stages with 1-D bulk TMA copies; cached rows never depend on the
//     previous kernel, so the first tiles are in flight before
//     griddepcontrol.wait;
//   * the new token's K/V (already rotated by the QKV kernel) are stored in the
//     cache format (fp32, fp16 round-to-nearest, or int8 with one fp16 scale
//     per row, k2-burn README "KV cache storage") by the CTA whose range holds
//     position pos, which also uses the stored values itself: no CTA reads a
//     row another CTA writes in the same launch;
//   * int8 rows are dequantised inside the kernel (code * row scale), so no
//     dequantised copy of the history is ever materialised;
//   * fp32 online softmax per tile; each split writes (m, l, o) and the last
//     CTA of a KV head to finish (atomic counter, no spin) merges the splits
//     with their log-sum-exp weights and writes the head outputs.
#include <math.h>

#include <type_traits>

#include "k2_kernels.h"
#include "k2_common.cuh"

namespace k2 {

namespace {

template <typename KVT>
struct KVTraits;
template <>
struct KVTraits<float> {
  static constexpr bool kI8 = false;
};
template <>
struct KVTraits<__half> {
  static constexpr bool kI8 = false;
};
template <>
struct KVTraits<int8_t> {
  static constexpr bool kI8 = true;
};

__device__ __forceinline__ float2 load2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 load2(const __half* p) {
  return __half22float2(*reinterpret_cast<const __half2*>(p));
}
__device__ __forceinline__ float2 load2(const int8_t* p) {
  const char2 c = *reinterpret_cast<const char2*>(p);
  return make_float2(static_cast<float>(c.x), static_cast<float>(c.y));
}

template <int D, int REP, typename KVT>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnArgs a) {
  constexpr int TK = kAttnTK;
  constexpr int ELT = sizeof(KVT);
  constexpr int EPL = 16 / ELT;  // elements per 16-byte load
  constexpr int LPK = D / EPL;   // lanes that share one key row
  static_assert(LPK >= 1 && LPK <= 32 && (32 % LPK) == 0, "head_dim / dtype");
  constexpr int KPW = 32 / LPK;  // keys per warp per pass
  constexpr int KPP = KPW * (kAttnThreads / 32);
  constexpr int NPASS = (TK + KPP - 1) / KPP;
  constexpr bool I8 = KVTraits<KVT>::kI8;
  constexpr int DP = D / 2;
  static_assert(kAttnThreads % DP == 0, "head_dim");
  constexpr int KG = kAttnThreads / DP;  // key groups of the PV product
  constexpr uint32_t ROWB = D * ELT;
  constexpr uint32_t KV_TILE = TK * ROWB;

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[4];
  __shared__ float S[REP][TK];
  __shared__ float P[REP][TK];
  __shared__ float m_sh[REP], l_sh[REP], al_sh[REP];
  __shared__ float red[KG * REP * D];
  __shared__ __align__(16) KVT newkv[2][D];
  __shared__ __half newsc[2];
  __shared__ int last_sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z, g = blockIdx.y, sp = blockIdx.x, ns = gridDim.x;
  const int seq = a.seq0 + b;
  // seq_len was written two or more launches back (see pdl_trigger placement)
  const int pos = a.seq_len[seq];
  if (pos < 0 || pos >= a.cap) {
    if (tid == 0) atomicOr(a.guard, GUARD_POS);
    return;  // every CTA of the launch sees the same pos and leaves the same way
  }
  const int L = pos + 1;
  const int k0 = min(L, static_cast<int>((static_cast<long long>(L) * sp) / ns) & ~7);
  const int k1 = (sp == ns - 1) ? L : min(L, static_cast<int>((static_cast<long long>(L) * (sp + 1)) / ns) & ~7);
  const int ntile = k1 > k0 ? (k1 - k0 + TK - 1) / TK : 0;
  const size_t head_row = (static_cast<size_t>(seq) * a.nkv + g) * a.cap;
  const uint8_t* Kg = reinterpret_cast<const uint8_t*>(a.kc) + head_row * ROWB;
  const uint8_t* Vg = reinterpret_cast<const uint8_t*>(a.vc) + head_row * ROWB;
  const __half* KSg = I8 ? reinterpret_cast<const __half*>(a.ks) + head_row : nullptr;
  const __half* VSg = I8 ? reinterpret_cast<const __half*>(a.vs) + head_row : nullptr;

  auto issue = [&](int t) {
    const int buf = t % a.nstage;
    uint8_t* stg = smem + static_cast<size_t>(buf) * a.stage_bytes;
    const int j0 = k0 + t * TK;
    const int rows = min(TK, k1 - j0);
    const int crow = max(0, min(rows, pos - j0));  // cached rows; row pos is the new one
    const int srow = (crow + 7) & ~7;             // scale copies in 16-byte units
    uint32_t bytes = 2u * crow * ROWB + (I8 && crow > 0 ? 2u * srow * 2u : 0u);
    if (bytes == 0) {
      mbar_arrive(&full[buf]);
      return;
    }
    mbar_arrive_expect_tx(&full[buf], bytes);
    bulk_g2s(stg, Kg + static_cast<size_t>(j0) * ROWB, crow * ROWB, &full[buf]);
    bulk_g2s(stg + KV_TILE, Vg + static_cast<size_t>(j0) * ROWB, crow * ROWB, &full[buf]);
    if constexpr (I8) {
      bulk_g2s(stg + 2 * KV_TILE, KSg + j0, srow * 2u, &full[buf]);
      bulk_g2s(stg + 2 * KV_TILE + TK * 2, VSg + j0, srow * 2u, &full[buf]);
    }
  };

  if (tid == 0) {
    for (int i = 0; i < a.nstage; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
    const int pre = min(a.nstage, ntile);
    for (int t = 0; t < pre; ++t) issue(t);
  }
  if (tid < REP) {
    m_sh[tid] = -INFINITY;
    l_sh[tid] = 0.f;
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  // ---- query slice (pre-scaled by 1/sqrt(D)) --------------------------------------
  const int kl = lane % LPK;
  const float* qkv = a.qkv + static_cast<size_t>(b) * a.qkv_stride;
  float q[REP][EPL];
#pragma unroll
  for (int h = 0; h < REP; ++h)
#pragma unroll
    for (int e = 0; e < EPL; ++e) q[h][e] = qkv[(g * REP + h) * D + kl * EPL + e] * a.scale;

  // ---- the new token's K/V in cache format ------------------------------------------
  const bool has_new = ntile > 0 && k1 == L;
  if (has_new && warp < 2) {
    const float* src = qkv + (warp == 0 ? a.nq * D : (a.nq + a.nkv) * D) + g * D;
    KVT* dst = reinterpret_cast<KVT*>(warp == 0 ? a.kc_w : a.vc_w) + (head_row + pos) * D;
    if constexpr (I8) {
      float amax = 0.f;
      for (int i = lane; i < D; i += 32) amax = fmaxf(amax, fabsf(src[i]));
      amax = warp_max(amax);
      const __half sh = __float2half_rn(fminf(amax / 127.0f, 65504.0f));
      const float sf = __half2float(sh);
      for (int i = lane; i < D; i += 32) {
        float c = sf > 0.f ? rintf(src[i] / sf) : 0.f;
        c = fminf(fmaxf(c, -127.f), 127.f);
        const int8_t ci = static_cast<int8_t>(c);
        dst[i] = ci;
        newkv[warp][i] = ci;
      }
      if (lane == 0) {
        (warp == 0 ? reinterpret_cast<__half*>(a.ks) : reinterpret_cast<__half*>(a.vs))[head_row + pos] = sh;
        newsc[warp] = sh;
      }
    } else if constexpr (std::is_same<KVT, __half>::value) {
      for (int i = lane; i < D; i += 32) {
        const __half hv = __float2half_rn(src[i]);
        dst[i] = hv;
        newkv[warp][i] = hv;
      }
    } else {
      for (int i = lane; i < D; i += 32) {
        dst[i] = src[i];
        newkv[warp][i] = src[i];
      }
    }
  }

  // ---- tiles ----------------------------------------------------------------------------
  const int kg = tid / DP, dp = tid % DP;
  float acc[REP][2];
#pragma unroll
  for (int h = 0; h < REP; ++h) acc[h][0] = acc[h][1] = 0.f;

  int t = 0;
  bool timed_out = false;
  for (; t < ntile; ++t) {
    const int buf = t % a.nstage;
    const uint32_t par = static_cast<uint32_t>(t / a.nstage) & 1u;
    const bool ok = mbar_wait(&full[buf], par);
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      break;
    }
    uint8_t* stg = smem + static_cast<size_t>(buf) * a.stage_bytes;
    const __half* ksc = reinterpret_cast<const __half*>(stg + 2 * KV_TILE);
    const __half* vsc = ksc + TK;
    const int j0 = k0 + t * TK;
    const int rows = min(TK, k1 - j0);
    if (has_new && pos >= j0 && pos < j0 + rows) {
      const int jr = pos - j0;
      if (tid < D) {
        reinterpret_cast<KVT*>(stg + jr * ROWB)[tid] = newkv[0][tid];
        reinterpret_cast<KVT*>(stg + KV_TILE + jr * ROWB)[tid] = newkv[1][tid];
      }
      if constexpr (I8) {
        if (tid == 0) {
          reinterpret_cast<__half*>(stg + 2 * KV_TILE)[jr] = newsc[0];
          reinterpret_cast<__half*>(stg + 2 * KV_TILE + TK * 2)[jr] = newsc[1];
        }
      }
      __syncthreads();
    }
    // scores
#pragma unroll
    for (int pass = 0; pass < NPASS; ++pass) {
      const int jj = pass * KPP + warp * KPW + lane / LPK;
      float dot[REP];
#pragma unroll
      for (int h = 0; h < REP; ++h) dot[h] = 0.f;
      if (jj < rows) {
        const uint4 v = *reinterpret_cast<const uint4*>(stg + jj * ROWB + kl * 16);
        float kf[EPL];
        Unpack<KVT>::run(v, kf);
#pragma unroll
        for (int h = 0; h < REP; ++h)
#pragma unroll
          for (int e = 0; e < EPL; ++e) dot[h] = fmaf(q[h][e], kf[e], dot[h]);
      }
#pragma unroll
      for (int h = 0; h < REP; ++h)
#pragma unroll
        for (int o = LPK / 2; o > 0; o >>= 1) dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], o);
      if (kl == 0 && jj < rows) {
        const float sc = I8 ? __half2float(ksc[jj]) : 1.f;
#pragma unroll
        for (int h = 0; h < REP; ++h) S[h][jj] = dot[h] * sc;
      }
    }
    __syncthreads();
    // online softmax, one warp per query head
    if (warp < REP) {
      const int h = warp;
      float mt = -INFINITY;
      for (int j = lane; j < rows; j += 32) mt = fmaxf(mt, S[h][j]);
      mt = warp_max(mt);
      const float mo = m_sh[h];
      const float mn = fmaxf(mo, mt);
      float sum = 0.f;
      for (int j = lane; j < rows; j += 32) {
        const float p = expf(S[h][j] - mn);
        sum += p;
        P[h][j] = I8 ? p * __half2float(vsc[j]) : p;
      }
      sum = warp_sum(sum);
      if (lane == 0) {
        const float al = expf(mo - mn);
        al_sh[h] = al;
        l_sh[h] = l_sh[h] * al + sum;
        m_sh[h] = mn;
      }
    }
    __syncthreads();
    // o = alpha * o + P . V
    {
      const KVT* vt = reinterpret_cast<const KVT*>(stg + KV_TILE);
#pragma unroll
      for (int h = 0; h < REP; ++h) {
        acc[h][0] *= al_sh[h];
        acc[h][1] *= al_sh[h];
      }
      for (int j = kg; j < rows; j += KG) {
        const float2 v = load2(vt + j * D + 2 * dp);
#pragma unroll
        for (int h = 0; h < REP; ++h) {
          const float p = P[h][j];
          acc[h][0] = fmaf(p, v.x, acc[h][0]);
          acc[h][1] = fmaf(p, v.y, acc[h][1]);
        }
      }
    }
    __syncthreads();
    if (tid == 0 && t + a.nstage < ntile) {
      fence_proxy_async();
      issue(t + a.nstage);
    }
  }

  if (timed_out) {
    if (tid == 0) {
      atomicOr(a.guard, GUARD_TIMEOUT);
      const int issued = min(ntile, t + a.nstage);
      for (int t2 = t; t2 < issued; ++t2)
        (void)mbar_wait(&full[t2 % a.nstage], static_cast<uint32_t>(t2 / a.nstage) & 1u);
    }
    __syncthreads();
  }

  // ---- this split's (m, l, o) ---------------------------------------------------------------
#pragma unroll
  for (int h = 0; h < REP; ++h) {
    red[(kg * REP + h) * D + 2 * dp] = acc[h][0];
    red[(kg * REP + h) * D + 2 * dp + 1] = acc[h][1];
  }
  __syncthreads();
  constexpr int PSTRIDE = REP * (D + 2);
  float* pp = a.part + ((static_cast<size_t>(b) * a.nkv + g) * ns + sp) * PSTRIDE;
  for (int idx = tid; idx < REP * D; idx += kAttnThreads) {
    const int h = idx / D, dim = idx - h * D;
    float o = 0.f;
    for (int q2 = 0; q2 < KG; ++q2) o += red[(q2 * REP + h) * D + dim];
    pp[2 * REP + idx] = o;
  }
  if (tid < REP) {
    pp[tid] = m_sh[tid];
    pp[REP + tid] = l_sh[tid];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&a.counter[b * a.nkv + g], 1u);
    last_sh = (prev == static_cast<unsigned>(ns - 1));
  }
  __syncthreads();
  if (!last_sh) return;

  // ---- last CTA of this KV head: log-sum-exp merge of the splits -------------------------------
  __threadfence();
  const float* base = a.part + (static_cast<size_t>(b) * a.nkv + g) * ns * PSTRIDE;
  for (int idx = tid; idx < REP * D; idx += kAttnThreads) {
    const int h = idx / D;
    float M = -INFINITY;
    for (int s2 = 0; s2 < ns; ++s2) M = fmaxf(M, __ldcg(base + s2 * PSTRIDE + h));
    float Ls = 0.f, O = 0.f;
    for (int s2 = 0; s2 < ns; ++s2) {
      const float ms = __ldcg(base + s2 * PSTRIDE + h);
      const float w = ms == -INFINITY ? 0.f : expf(ms - M);
      Ls = fmaf(__ldcg(base + s2 * PSTRIDE + REP + h), w, Ls);
      O = fmaf(__ldcg(base + s2 * PSTRIDE + 2 * REP + idx), w, O);
    }
    a.out[static_cast<size_t>(b) * a.nq * D + (g * REP + h) * D + (idx - h * D)] = O / Ls;
  }
  if (tid == 0) a.counter[b * a.nkv + g] = 0u;
}

template <int D, int REP>
cudaError_t launch_dr(const AttnArgs& a, int kv_dtype, const cudaLaunchConfig_t& cfg) {
  switch (kv_dtype) {
    case 0: return cudaLaunchKernelEx(&cfg, attn_decode_kernel<D, REP, float>, a);
    case 2: return cudaLaunchKernelEx(&cfg, attn_decode_kernel<D, REP, __half>, a);
    case 3: return cudaLaunchKernelEx(&cfg, attn_decode_kernel<D, REP, int8_t>, a);
  }
  return cudaErrorInvalidValue;
}

template <int D, int REP>
cudaError_t attr_dr(int bytes) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(attn_decode_kernel<D, REP, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)))
    return e;
  if ((e = cudaFuncSetAttribute(attn_decode_kernel<D, REP, __half>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)))
    return e;
  return cudaFuncSetAttribute(attn_decode_kernel<D, REP, int8_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

#define K2_ATTN_SHAPES(X) \
  X(16, 1) X(16, 2) X(16, 4) X(64, 1) X(64, 2) X(64, 4) X(128, 1) X(128, 2) X(128, 4)

}  // namespace

bool attn_supported(int head_dim, int rep, int kv_dtype) {
  if (kv_dtype != 0 && kv_dtype != 2 && kv_dtype != 3) return false;
#define K2_ATTN_SUP(D, R) \
  if (head_dim == D && rep == R) return true;
  K2_ATTN_SHAPES(K2_ATTN_SUP)
#undef K2_ATTN_SUP
  return false;
}

size_t attn_stage_bytes(int head_dim, int kv_dtype) {
  const size_t elt = kv_dtype == 0 ? 4 : (kv_dtype == 2 ? 2 : 1);
  return 2 * kAttnTK * head_dim * elt + (kv_dtype == 3 ? 2 * kAttnTK * 2 : 0);
}

cudaError_t attn_init_attrs() {
  cudaError_t e = cudaSuccess;
#define K2_ATTN_ATTR(D, R) \
  if (e == cudaSuccess) e = attr_dr<D, R>(160 * 1024);
  K2_ATTN_SHAPES(K2_ATTN_ATTR)
#undef K2_ATTN_ATTR
  return e;
}

cudaError_t launch_attn(const AttnArgs& a, int head_dim, int rep, int kv_dtype, int nsplit, int batch,
                        cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nsplit, a.nkv, batch);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(a.nstage) * a.stage_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
#define K2_ATTN_LAUNCH(D, R) \
  if (head_dim == D && rep == R) return launch_dr<D, R>(a, kv_dtype, cfg);
  K2_ATTN_SHAPES(K2_ATTN_LAUNCH)
#undef K2_ATTN_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace k2
