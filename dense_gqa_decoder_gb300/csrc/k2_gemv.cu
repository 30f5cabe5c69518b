// Streaming GEMV for batch-1 decode: y = W . norm(x), with the epilogue of the
// step it serves fused in.
//
// The decode step is bound by HBM: every weight byte is read once per token
// and used for one multiply-add (k2-burn README, "Model shape": 8.8 GB of bf16
// weights per token for the 3.7B shape).  So the kernel is built to keep bytes
// in flight, not to do arithmetic:
//   * one CTA per SM owns a contiguous band of rows; an elected thread streams
//     the band through a ring of shared-memory stages with 1-D bulk TMA copies
//     (cp.async.bulk + mbarrier complete_tx), several stages ahead;
//   * the first stages are issued before griddepcontrol.wait, i.e. while the
//     previous kernel of the step is still finishing (weights never depend on
//     it), which hides the ramp-up of each launch;
//   * each lane keeps its slice of the (normalised) input vector in registers
//     and reads weights from shared memory with 128-bit loads; a warp owns one
//     (row, K-slice) pair per stage and reduces with shuffles;
//   * the norm of the input (GroupedRMSNorm, k2-burn README "Status: v0") is
//     computed in the prologue of the consuming GEMV from the fp32 residual
//     stream, so it never makes a separate pass over HBM;
//   * epilogues: residual add (o_proj, down_proj), split-half RoPE on row pairs
//     (QKV, rows repacked so that i and i + d/2 of a head are adjacent),
//     SwiGLU on interleaved gate/up rows, and lm_head logits with a fused
//     first-index argmax (kimi-k3-in-c k3_run.c, `argmax_`).
#include <math.h>

#include "k2_kernels.h"
#include "k2_common.cuh"

namespace k2 {

namespace {

struct BestPair {
  float v;
  int i;
};

// first index of the maximum: larger value wins, equal values go to the lower index
__device__ __forceinline__ BestPair better(BestPair a, BestPair b) {
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}

__device__ __forceinline__ BestPair warp_best(BestPair p) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    BestPair q;
    q.v = __shfl_xor_sync(0xffffffffu, p.v, o);
    q.i = __shfl_xor_sync(0xffffffffu, p.i, o);
    p = better(p, q);
  }
  return p;
}

template <typename WT, int EPI>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_kernel(const GemvArgs a) {
  constexpr int EPL = Unpack<WT>::N;  // weights per 16-byte load
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[8];
  __shared__ float red[2][8][8];  // [stage parity][row in stage][slice]
  __shared__ float ss_sh[8][4];   // [slice][group] sums of squares
  __shared__ float rs_sh[4];      // 1 / rms per group
  __shared__ BestPair best_sh[8];
  __shared__ int last_sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int units = a.N / a.align;
  const int r0 = static_cast<int>((static_cast<long long>(units) * cta) / G) * a.align;
  const int r1 = static_cast<int>((static_cast<long long>(units) * (cta + 1)) / G) * a.align;
  const int nrows = r1 - r0;
  const int nst = (nrows + a.R - 1) / a.R;
  const size_t row_bytes = static_cast<size_t>(a.K) * sizeof(WT);
  const uint8_t* Wb = reinterpret_cast<const uint8_t*>(a.W);

  auto issue = [&](int st) {
    const int buf = st % a.nstage;
    const int rows = min(a.R, nrows - st * a.R);
    const uint32_t bytes = static_cast<uint32_t>(rows * row_bytes);
    mbar_arrive_expect_tx(&full[buf], bytes);
    bulk_g2s(smem + static_cast<size_t>(buf) * a.stage_bytes,
             Wb + static_cast<size_t>(r0 + st * a.R) * row_bytes, bytes, &full[buf]);
  };

  // ---- prologue: start streaming weights before the previous kernel is done
  if (tid == 0) {
    for (int i = 0; i < a.nstage; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
    const int pre = min(a.nstage, nst);
    for (int st = 0; st < pre; ++st) issue(st);
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  // ---- this lane's slice of x, normalised --------------------------------------
  const int sl = warp % a.nslice;
  const int rw = warp / a.nslice;
  float xr[kGemvKcMax][EPL];
#pragma unroll
  for (int c = 0; c < kGemvKcMax; ++c) {
    const int e0 = ((sl * a.kc + c) * 32 + lane) * EPL;
    const bool ok = c < a.kc && e0 < a.K;
#pragma unroll
    for (int j = 0; j < EPL; j += 4) {
      float4 v = ok ? __ldcg(reinterpret_cast<const float4*>(a.x + e0 + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
      xr[c][j] = v.x; xr[c][j + 1] = v.y; xr[c][j + 2] = v.z; xr[c][j + 3] = v.w;
    }
  }
  if (a.gain != nullptr) {
    const int gsz = a.K / a.groups;
    float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < kGemvKcMax; ++c) {
      const int e0 = ((sl * a.kc + c) * 32 + lane) * EPL;
      const int grp = e0 / gsz;
      float t = 0.f;
#pragma unroll
      for (int j = 0; j < EPL; ++j) t = fmaf(xr[c][j], xr[c][j], t);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q == grp) ss[q] += t;  // out-of-range chunks hold zeros
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) ss[q] = warp_sum(ss[q]);
    if (rw == 0 && lane == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) ss_sh[sl][q] = ss[q];
    }
    __syncthreads();
    if (tid < a.groups) {
      float t = 0.f;
      for (int q = 0; q < a.nslice; ++q) t += ss_sh[q][tid];
      rs_sh[tid] = 1.0f / sqrtf(t / static_cast<float>(gsz) + a.eps);
    }
    __syncthreads();
    const WT* gw = reinterpret_cast<const WT*>(a.gain);
#pragma unroll
    for (int c = 0; c < kGemvKcMax; ++c) {
      const int e0 = ((sl * a.kc + c) * 32 + lane) * EPL;
      if (c < a.kc && e0 < a.K) {
        const float r = rs_sh[e0 / gsz];
        float gf[EPL];
        Unpack<WT>::run(__ldg(reinterpret_cast<const uint4*>(gw + e0)), gf);
#pragma unroll
        for (int j = 0; j < EPL; ++j) xr[c][j] = xr[c][j] * r * gf[j];
      }
    }
  }

  // ---- main loop over the ring ----------------------------------------------------
  BestPair best{-INFINITY, 0x7fffffff};
  int st = 0;
  bool timed_out = false;
  for (; st < nst; ++st) {
    const int buf = st % a.nstage;
    const uint32_t par = static_cast<uint32_t>(st / a.nstage) & 1u;
    const bool ok = mbar_wait(&full[buf], par);
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      break;
    }
    const int rows = min(a.R, nrows - st * a.R);
    if (rw < rows) {
      const uint8_t* rowp = smem + static_cast<size_t>(buf) * a.stage_bytes + rw * row_bytes;
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int c = 0; c < kGemvKcMax; ++c) {
        const int e0 = ((sl * a.kc + c) * 32 + lane) * EPL;
        if (c < a.kc && e0 < a.K) {
          const uint4 v = *reinterpret_cast<const uint4*>(rowp + static_cast<size_t>(e0) * sizeof(WT));
          float w[EPL];
          Unpack<WT>::run(v, w);
          float t = 0.f;
#pragma unroll
          for (int j = 0; j < EPL; ++j) t = fmaf(w[j], xr[c][j], t);
          if (c & 1) acc1 += t; else acc0 += t;
        }
      }
      const float dsum = warp_sum(acc0 + acc1);
      if (lane == 0) red[st & 1][rw][sl] = dsum;
    }
    __syncthreads();
    if (tid == 0 && st + a.nstage < nst) {
      fence_proxy_async();
      issue(st + a.nstage);
    }
    // ---- epilogue of this stage
    const int row_base = r0 + st * a.R;
    if constexpr (EPI == EPI_QKV || EPI == EPI_SWIGLU) {
      if (tid < rows / 2) {
        float v0 = 0.f, v1 = 0.f;
        for (int q = 0; q < a.nslice; ++q) {
          v0 += red[st & 1][2 * tid][q];
          v1 += red[st & 1][2 * tid + 1][q];
        }
        const int P = row_base / 2 + tid;
        if constexpr (EPI == EPI_SWIGLU) {
          a.out[P] = v0 / (1.0f + expf(-v0)) * v1;
        } else {
          const int half = a.head_dim / 2;
          const int head = P / half, i = P - head * half;
          float o0 = v0, o1 = v1;
          if (head < a.n_rot_heads) {
            int pos = a.seq_len[a.seq];
            if (pos < 0 || pos >= a.cap) {
              atomicOr(a.guard, GUARD_POS);
              pos = 0;
            }
            const float2 cs = a.rope[static_cast<size_t>(pos) * half + i];
            o0 = v0 * cs.x - v1 * cs.y;
            o1 = v1 * cs.x + v0 * cs.y;
          }
          a.out[head * a.head_dim + i] = o0;
          a.out[head * a.head_dim + i + half] = o1;
        }
      }
    } else {
      if (tid < rows) {
        float v = 0.f;
        for (int q = 0; q < a.nslice; ++q) v += red[st & 1][tid][q];
        const int row = row_base + tid;
        if constexpr (EPI == EPI_STORE) {
          a.out[row] = v;
        } else if constexpr (EPI == EPI_RESID) {
          a.out[row] += v;
        } else {
          if (a.logits) a.logits[row] = v;
          if (v != v) atomicOr(a.guard, GUARD_NAN);
          else best = better(best, BestPair{v, row});
        }
      }
    }
  }

  if (timed_out) {
    if (tid == 0) {
      atomicOr(a.guard, GUARD_TIMEOUT);
      // let the copies still in flight land before this CTA's shared memory is released
      const int issued = min(nst, st + a.nstage);
      for (int s2 = st; s2 < issued; ++s2)
        (void)mbar_wait(&full[s2 % a.nstage], static_cast<uint32_t>(s2 / a.nstage) & 1u);
    }
    __syncthreads();
  }

  if constexpr (EPI == EPI_ARGMAX) {
    best = warp_best(best);
    if (lane == 0) best_sh[warp] = best;
    __syncthreads();
    if (tid == 0) {
      BestPair b = best_sh[0];
      for (int w = 1; w < kGemvThreads / 32; ++w) b = better(b, best_sh[w]);
      a.part_val[cta] = b.v;
      a.part_idx[cta] = b.i;
      __threadfence();
      const unsigned t = atomicAdd(a.counter, 1u);
      last_sh = (t == static_cast<unsigned>(G - 1));
    }
    __syncthreads();
    if (last_sh) {
      __threadfence();
      // every CTA raised its guard bits before it counted itself, so the
      // last one sees them all; a timed-out CTA's partial maximum covers only
      // the rows that arrived, so no token comes out of such a launch
      const unsigned g = __ldcg(a.guard);
      const bool timed = (g & GUARD_TIMEOUT) != 0u;
      BestPair b{-INFINITY, 0x7fffffff};
      for (int i = tid; i < G; i += kGemvThreads) b = better(b, BestPair{__ldcg(a.part_val + i), __ldcg(a.part_idx + i)});
      b = warp_best(b);
      if (lane == 0) best_sh[warp] = b;
      __syncthreads();
      if (tid == 0) {
        BestPair f = best_sh[0];
        for (int w = 1; w < kGemvThreads / 32; ++w) f = better(f, best_sh[w]);
        bool nan = (g & GUARD_NAN) != 0u;
        if (f.i == 0x7fffffff) {  // every logit was NaN
          atomicOr(a.guard, GUARD_NAN);
          f.i = 0;
          nan = true;
        }
        if (a.fail_token) {
          *a.next_token = (nan || timed) ? -1 : f.i;
        } else if (!timed) {
          *a.next_token = f.i;
          if (a.advance) a.seq_len[a.seq] += 1;
        }
        *a.counter = 0u;
      }
    }
  }
}

template <typename WT>
cudaError_t launch_typed(const GemvArgs& a, int epi, const cudaLaunchConfig_t& cfg) {
  switch (epi) {
    case EPI_STORE: return cudaLaunchKernelEx(&cfg, gemv_kernel<WT, EPI_STORE>, a);
    case EPI_RESID: return cudaLaunchKernelEx(&cfg, gemv_kernel<WT, EPI_RESID>, a);
    case EPI_QKV: return cudaLaunchKernelEx(&cfg, gemv_kernel<WT, EPI_QKV>, a);
    case EPI_SWIGLU: return cudaLaunchKernelEx(&cfg, gemv_kernel<WT, EPI_SWIGLU>, a);
    case EPI_ARGMAX: return cudaLaunchKernelEx(&cfg, gemv_kernel<WT, EPI_ARGMAX>, a);
  }
  return cudaErrorInvalidValue;
}

template <typename WT>
cudaError_t set_smem_attr(size_t bytes) {
  cudaError_t e = cudaSuccess;
  const int b = static_cast<int>(bytes);
  if ((e = set_kernel_smem(gemv_kernel<WT, EPI_STORE>, b))) return e;
  if ((e = set_kernel_smem(gemv_kernel<WT, EPI_RESID>, b))) return e;
  if ((e = set_kernel_smem(gemv_kernel<WT, EPI_QKV>, b))) return e;
  if ((e = set_kernel_smem(gemv_kernel<WT, EPI_SWIGLU>, b))) return e;
  return set_kernel_smem(gemv_kernel<WT, EPI_ARGMAX>, b);
}

}  // namespace

bool gemv_plan(GemvArgs& a, int wbytes, int epi, size_t smem_budget) {
  if (wbytes != 2 && wbytes != 4) return false;
  const int EPL = 16 / wbytes;
  const int CH = 32 * EPL;
  if (a.N <= 0 || a.K <= 0 || a.K % EPL) return false;
  const size_t row_bytes = static_cast<size_t>(a.K) * wbytes;
  size_t r = 20480 / row_bytes;
  int R = static_cast<int>(r < 1 ? 1 : (r > 8 ? 8 : r));
  while (R & (R - 1)) R &= R - 1;  // power of two
  const bool pairs = (epi == EPI_QKV || epi == EPI_SWIGLU);
  if (pairs && R < 2) R = 2;
  if (pairs && (a.N % 2)) return false;
  const int nslice = 8 / R;
  const int CT = (a.K + CH - 1) / CH;
  const int kc = (CT + nslice - 1) / nslice;
  if (kc > kGemvKcMax) return false;
  if (a.gain) {
    if (a.groups < 1 || a.groups > 4 || a.K % a.groups || (a.K / a.groups) % EPL) return false;
  }
  a.R = R;
  a.nslice = nslice;
  a.kc = kc;
  a.align = pairs ? 2 : 1;
  a.stage_bytes = static_cast<uint32_t>(R * row_bytes);
  size_t ns = smem_budget / a.stage_bytes;
  if (ns > 8) ns = 8;
  if (ns < 2) return false;
  a.nstage = static_cast<int>(ns);
  return true;
}

size_t gemv_smem_bytes(const GemvArgs& a) { return static_cast<size_t>(a.nstage) * a.stage_bytes; }

cudaError_t gemv_init_attrs() {
  cudaError_t e = set_smem_attr<__nv_bfloat16>(200 * 1024);
  if (e != cudaSuccess) return e;
  return set_smem_attr<float>(200 * 1024);
}

cudaError_t launch_gemv(const GemvArgs& a, int wbytes, int epi, int grid, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = gemv_smem_bytes(a);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return wbytes == 2 ? launch_typed<__nv_bfloat16>(a, epi, cfg) : launch_typed<float>(a, epi, cfg);
}

}  // namespace k2
