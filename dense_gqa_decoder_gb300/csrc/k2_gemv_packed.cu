// Packed streaming GEMV: the batch-1 decode projections y = W . norm(x) with
// the epilogue of each step fused in (QKV + split-half RoPE, o_proj and
// down_proj + residual, gate/up + SwiGLU, lm_head + first-index argmax).
//
// The decode step is bound by HBM: each weight byte is read once per token for
// one multiply-add (k2-burn README, "Model shape": 8.8 GB of bf16 weights per
// token at the 3.7B shape).  Measured on this GPU, a read stream reaches about
// 7.2-7.5 TB/s either with many plain 128-bit loads in flight or with 1-D bulk
// TMA copies of at least 4 KB and about 64 KB in flight per SM; 1 KB copies
// stall near 3 TB/s.  The kernel is shaped by that:
//   * at set-up every matrix is packed pair-interleaved in 512-byte chunks:
//     [row pair][chunk][row 0 | row 1], zero-padded, so the (pair, chunk) units
//     of any contiguous range are one contiguous run of bytes (1 KB per unit);
//   * a CTA owns a band of row pairs; its units are cut into 8 equal
//     contiguous ranges, one per warp (exact balance for any shape); each warp
//     streams its range through its own ring of shared-memory slots with one
//     bulk copy of 4-5 KB per slot, refilled by lane 0 as soon as the warp has
//     read it: no CTA barrier inside the loop;
//   * the first slots are requested before griddepcontrol.wait, while the
//     previous kernel of the step is still finishing (weights never depend on
//     it);
//   * x is normalised once per CTA (GroupedRMSNorm, k2-burn README "Status:
//     v0") from the fp32 residual stream into shared memory, lane-interleaved
//     per chunk, so every 128-bit read of x and W is conflict-free and each x
//     chunk serves both rows of a pair;
//   * a pair is finished by the warp that read all of it; the few pairs cut by
//     a warp boundary are summed piece by piece in warp order at the end, so
//     results are deterministic.
#include <math.h>

#include "k2_kernels.h"
#include "k2_common.cuh"

namespace k2 {

namespace {

constexpr int kUnitB = 1024;  // one chunk of both rows of a pair

struct Best {
  float v;
  int i;
};
__device__ __forceinline__ Best better(Best a, Best b) {
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}
__device__ __forceinline__ Best warp_best(Best p) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Best q;
    q.v = __shfl_xor_sync(0xffffffffu, p.v, o);
    q.i = __shfl_xor_sync(0xffffffffu, p.i, o);
    p = better(p, q);
  }
  return p;
}

template <typename WT>
__device__ __forceinline__ float4 load_gain4(const void* g, int e);
template <>
__device__ __forceinline__ float4 load_gain4<__nv_bfloat16>(const void* g, int e) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(g) + e));
  return make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
}
template <>
__device__ __forceinline__ float4 load_gain4<float>(const void* g, int e) {
  return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(g) + e));
}

template <typename WT, int EPI>
__global__ void __launch_bounds__(kPackedThreads, 1) packed_gemv_kernel(const PackedGemvArgs a) {
  constexpr int EPL = Unpack<WT>::N;  // elements per 16-byte load
  constexpr int CH = 32 * EPL;        // elements per chunk
  constexpr int NPL = EPL / 4;        // float4 planes of x per chunk
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[kPackedWarps][kPackedMaxSlots];
  __shared__ float ss_sh[kPackedWarps][4];
  __shared__ float rs_sh[4];
  __shared__ int rec_pair[kPackedWarps][2];
  __shared__ float rec_val[kPackedWarps][2][2];
  __shared__ int rec_n[kPackedWarps];
  __shared__ Best best_sh[kPackedWarps];
  __shared__ int last_sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int CT = a.CT, K = a.K, SU = a.SU, NS = a.NS;
  const int npairs = (a.N + 1) / 2;
  const int p0 = static_cast<int>((static_cast<long long>(npairs) * cta) / G);
  const int p1 = static_cast<int>((static_cast<long long>(npairs) * (cta + 1)) / G);
  const long long U = static_cast<long long>(p1 - p0) * CT;
  const int ua = static_cast<int>((U * warp) / kPackedWarps);
  const int ub = static_cast<int>((U * (warp + 1)) / kPackedWarps);
  const int nslots = (ub - ua + SU - 1) / SU;
  const uint8_t* src = reinterpret_cast<const uint8_t*>(a.Wp) + static_cast<size_t>(p0) * CT * kUnitB;
  uint8_t* ring = smem + static_cast<size_t>(warp) * NS * SU * kUnitB;
  float* xs = reinterpret_cast<float*>(smem + static_cast<size_t>(kPackedWarps) * NS * SU * kUnitB);

  auto issue = [&](int k) {
    const int u0 = ua + k * SU;
    const int n = min(SU, ub - u0);
    const int slot = k % NS;
    mbar_arrive_expect_tx(&full[warp][slot], static_cast<uint32_t>(n) * kUnitB);
    bulk_g2s(ring + static_cast<size_t>(slot) * SU * kUnitB, src + static_cast<size_t>(u0) * kUnitB,
             static_cast<uint32_t>(n) * kUnitB, &full[warp][slot]);
  };

  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&full[warp][i], 1);
    fence_mbar_init();
    for (int k = 0; k < NS && k < nslots; ++k) issue(k);
    rec_n[warp] = 0;
  }
  // norm gains are weights: fetch them before waiting for the previous kernel
  constexpr int PG = 4;   // float4s of the gain per thread kept in registers (K <= 4096)
  constexpr int PX = 10;  // float4s of x per thread loaded at once (K <= 10240)
  const int KP = CT * CH;
  const int gsz = a.gain ? K / a.groups : K;
  float4 gq[PG];
#pragma unroll
  for (int i = 0; i < PG; ++i) {
    const int e = tid * 4 + i * kPackedThreads * 4;
    gq[i] = (a.gain != nullptr && e < K) ? load_gain4<WT>(a.gain, e) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncwarp();
  pdl_wait();

  // ---- normalised x, lane-interleaved per chunk, zero past K ---------------------
  // All loads of x are issued before any is used: one L2 round trip.
  {
    auto xidx = [&](int e) {
      const int c = e / CH, r = e - c * CH, l = r / EPL, j = r - l * EPL;
      return ((c * NPL + j / 4) * 32 + l) * 4;
    };
    float ssq[4] = {0.f, 0.f, 0.f, 0.f};
    auto add_ssq = [&](int e, float4 v) {
      const float t = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      const int grp = e < K ? e / gsz : 4;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q == grp) ssq[q] += t;
    };
    float4 xq[PX];
#pragma unroll
    for (int i = 0; i < PX; ++i) {
      const int e = tid * 4 + i * kPackedThreads * 4;
      xq[i] = e < K ? __ldcg(reinterpret_cast<const float4*>(a.x + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < PX; ++i) add_ssq(tid * 4 + i * kPackedThreads * 4, xq[i]);
    for (int e = tid * 4 + PX * kPackedThreads * 4; e < KP; e += kPackedThreads * 4) {
      const float4 v = e < K ? __ldcg(reinterpret_cast<const float4*>(a.x + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(xs + xidx(e)) = v;
      add_ssq(e, v);
    }
    if (a.gain != nullptr) {
#pragma unroll
      for (int q = 0; q < 4; ++q) ssq[q] = warp_sum(ssq[q]);
      if (lane == 0)
        for (int q = 0; q < 4; ++q) ss_sh[warp][q] = ssq[q];
      __syncthreads();
      if (tid < a.groups) {
        float t = 0.f;
        for (int w = 0; w < kPackedWarps; ++w) t += ss_sh[w][tid];
        rs_sh[tid] = 1.0f / sqrtf(t / static_cast<float>(gsz) + a.eps);
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < PX; ++i) {
        const int e = tid * 4 + i * kPackedThreads * 4;
        if (e < KP) {
          float4 v = xq[i];
          if (e < K) {
            const float rs = rs_sh[e / gsz];
            const float4 gn = i < PG ? gq[i < PG ? i : 0] : load_gain4<WT>(a.gain, e);
            v.x = v.x * rs * gn.x; v.y = v.y * rs * gn.y; v.z = v.z * rs * gn.z; v.w = v.w * rs * gn.w;
          }
          *reinterpret_cast<float4*>(xs + xidx(e)) = v;
        }
      }
      for (int e = tid * 4 + PX * kPackedThreads * 4; e < K; e += kPackedThreads * 4) {
        float4* p = reinterpret_cast<float4*>(xs + xidx(e));
        const float rs = rs_sh[e / gsz];
        const float4 gn = load_gain4<WT>(a.gain, e);
        float4 v = *p;
        v.x = v.x * rs * gn.x; v.y = v.y * rs * gn.y; v.z = v.z * rs * gn.z; v.w = v.w * rs * gn.w;
        *p = v;
      }
    } else {
#pragma unroll
      for (int i = 0; i < PX; ++i) {
        const int e = tid * 4 + i * kPackedThreads * 4;
        if (e < KP) *reinterpret_cast<float4*>(xs + xidx(e)) = xq[i];
      }
    }
    __syncthreads();
  }
  // the next kernel may start its weight prefetch now that this one's reads
  // of the previous kernel's output are done
  pdl_trigger();

  // ---- epilogue of one finished pair (lane 0 / thread 0) ----------------------------
  Best best{-INFINITY, 0x7fffffff};
  auto finish = [&](int g, float v0, float v1) {
    const int row = 2 * g;
    if constexpr (EPI == EPI_SWIGLU) {
      a.out[g] = v0 / (1.0f + expf(-v0)) * v1;
    } else if constexpr (EPI == EPI_QKV) {
      const int half = a.head_dim / 2;
      const int head = g / half, i = g - head * half;
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
    } else {
      const int rows = min(2, a.N - row);
      const float v[2] = {v0, v1};
      for (int r = 0; r < rows; ++r) {
        if constexpr (EPI == EPI_STORE) {
          a.out[row + r] = v[r];
        } else if constexpr (EPI == EPI_RESID) {
          a.out[row + r] += v[r];
        } else {
          if (a.logits) a.logits[row + r] = v[r];
          if (v[r] != v[r]) atomicOr(a.guard, GUARD_NAN);
          else best = better(best, Best{v[r], row + r});
        }
      }
    }
  };

  // ---- stream this warp's units ---------------------------------------------------------
  int pl = ua / CT, c = ua - (ua / CT) * CT;  // current pair (CTA-local) and chunk
  bool pair_whole = (c == 0);                 // this warp saw the pair from its first chunk
  float acc0 = 0.f, acc1 = 0.f;
  bool bad = false;
  int k = 0;
  for (; k < nslots; ++k) {
    const int slot = k % NS;
    const bool ok = mbar_wait(&full[warp][slot], static_cast<uint32_t>(k / NS) & 1u);
    if (__any_sync(0xffffffffu, !ok)) {
      bad = true;
      break;
    }
    const uint8_t* buf = ring + static_cast<size_t>(slot) * SU * kUnitB;
    const int u0 = ua + k * SU;
    const int n = min(SU, ub - u0);
    int j = 0;
    while (j < n) {
      const int seg = min(n - j, CT - c);  // units of the current pair in this slot
#pragma unroll 2
      for (int q = 0; q < seg; ++q) {
        const int cc = c + q;
        float xv[EPL];
#pragma unroll
        for (int p = 0; p < NPL; ++p) {
          const float4 t = *reinterpret_cast<const float4*>(xs + ((cc * NPL + p) * 32 + lane) * 4);
          xv[4 * p] = t.x; xv[4 * p + 1] = t.y; xv[4 * p + 2] = t.z; xv[4 * p + 3] = t.w;
        }
        const uint8_t* ub8 = buf + (j + q) * kUnitB + lane * 16;
        float w0[EPL], w1[EPL];
        Unpack<WT>::run(*reinterpret_cast<const uint4*>(ub8), w0);
        Unpack<WT>::run(*reinterpret_cast<const uint4*>(ub8 + 512), w1);
        float t0 = 0.f, t1 = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          t0 = fmaf(w0[e], xv[e], t0);
          t1 = fmaf(w1[e], xv[e], t1);
        }
        acc0 += t0;
        acc1 += t1;
      }
      j += seg;
      c += seg;
      const bool pair_end = (c == CT);
      const bool range_end = (u0 + j == ub);
      if (pair_end || range_end) {
        const float s0 = warp_sum(acc0), s1 = warp_sum(acc1);
        acc0 = acc1 = 0.f;
        if (lane == 0) {
          if (pair_whole && pair_end) {
            finish(p0 + pl, s0, s1);
          } else {  // a piece of a pair cut by a warp boundary
            const int r = rec_n[warp];
            rec_pair[warp][r] = pl;
            rec_val[warp][r][0] = s0;
            rec_val[warp][r][1] = s1;
            rec_n[warp] = r + 1;
          }
        }
        if (pair_end) {
          ++pl;
          c = 0;
          pair_whole = true;
        }
      }
    }
    __syncwarp();
    if (lane == 0 && k + NS < nslots) {
      fence_proxy_async();
      issue(k + NS);
    }
  }

  if (bad && lane == 0) {
    atomicOr(a.guard, GUARD_TIMEOUT);
    // let the copies still in flight land before shared memory is released
    const int issued = min(nslots, k + NS);
    for (int k2 = k; k2 < issued; ++k2)
      (void)mbar_wait(&full[warp][k2 % NS], static_cast<uint32_t>(k2 / NS) & 1u);
  }
  __syncthreads();

  // ---- pairs cut by warp boundaries: pieces summed in warp order ------------------------
  if (tid == 0) {
    int cur = -1;
    float v0 = 0.f, v1 = 0.f;
    for (int w = 0; w < kPackedWarps; ++w) {
      for (int r = 0; r < rec_n[w]; ++r) {
        if (rec_pair[w][r] != cur) {
          if (cur >= 0) finish(p0 + cur, v0, v1);
          cur = rec_pair[w][r];
          v0 = v1 = 0.f;
        }
        v0 += rec_val[w][r][0];
        v1 += rec_val[w][r][1];
      }
    }
    if (cur >= 0) finish(p0 + cur, v0, v1);
  }

  if constexpr (EPI == EPI_ARGMAX) {
    best = warp_best(best);
    if (lane == 0) best_sh[warp] = best;
    __syncthreads();
    if (tid == 0) {
      Best b = best_sh[0];
      for (int w = 1; w < kPackedWarps; ++w) b = better(b, best_sh[w]);
      a.part_val[cta] = b.v;
      a.part_idx[cta] = b.i;
      __threadfence();
      const unsigned t = atomicAdd(a.counter, 1u);
      last_sh = (t == static_cast<unsigned>(G - 1));
    }
    __syncthreads();
    if (last_sh) {
      __threadfence();
      // a timed-out CTA's partial maximum covers only the rows that arrived:
      // such a launch writes no token and leaves the sequence where it was
      const bool timed = (__ldcg(a.guard) & GUARD_TIMEOUT) != 0u;
      Best b{-INFINITY, 0x7fffffff};
      for (int i = tid; i < G; i += kPackedThreads) b = better(b, Best{__ldcg(a.part_val + i), __ldcg(a.part_idx + i)});
      b = warp_best(b);
      if (lane == 0) best_sh[warp] = b;
      __syncthreads();
      if (tid == 0) {
        Best f = best_sh[0];
        for (int w = 1; w < kPackedWarps; ++w) f = better(f, best_sh[w]);
        if (f.i == 0x7fffffff) {  // every logit was NaN
          atomicOr(a.guard, GUARD_NAN);
          f.i = 0;
        }
        if (!timed) {
          *a.next_token = f.i;
          if (a.advance) a.seq_len[a.seq] += 1;
        }
        *a.counter = 0u;
      }
    }
  }
}

// ---- packing (set-up) ----------------------------------------------------------------------
// The source row of packed row R (null past N), per PackMode.
template <typename WT>
__device__ __forceinline__ const WT* pack_src_row(const WT* s0, const WT* s1, const WT* s2, int mode, int R, int N,
                                                  int K, int nq, int nkv, int d) {
  if (R >= N) return nullptr;
  if (mode == PACK_PLAIN) return s0 + static_cast<size_t>(R) * K;
  if (mode == PACK_GATEUP) return ((R & 1) ? s1 : s0) + static_cast<size_t>(R >> 1) * K;
  const int head = R / d, rr = R - head * d;
  const int sr = (rr & 1) ? (rr >> 1) + d / 2 : (rr >> 1);
  if (head < nq) return s0 + (static_cast<size_t>(head) * d + sr) * K;
  if (head < nq + nkv) return s1 + (static_cast<size_t>(head - nq) * d + sr) * K;
  return s2 + (static_cast<size_t>(head - nq - nkv) * d + sr) * K;
}

template <typename WT>
__global__ void pack_kernel(WT* __restrict__ dst, const WT* __restrict__ s0, const WT* __restrict__ s1,
                            const WT* __restrict__ s2, int mode, int N, int K, int CT, int nq, int nkv, int d) {
  constexpr int CH = 512 / sizeof(WT);
  const int R = blockIdx.x;  // packed row index (2 * pair + r)
  const int pair = R >> 1, r = R & 1;
  const WT* src = pack_src_row(s0, s1, s2, mode, R, N, K, nq, nkv, d);
  WT* out = dst + static_cast<size_t>(pair) * CT * 2 * CH + r * CH;
  for (int e = threadIdx.x; e < CT * CH; e += blockDim.x) {
    const int c = e / CH, i = e - c * CH;
    out[static_cast<size_t>(c) * 2 * CH + i] = (src != nullptr && e < K) ? src[e] : WT(0.f);
  }
}

// fp8 (E4M3) weight rows from bf16 (k2-burn README, "Post-training
// quantization": fp8 checkpoints the engine runs directly): per packed row
// (the row mapping of pack_kernel) s = max|w| / 448 and code = E4M3(w / s),
// nearest with ties to even, saturating; a zero row gets s = 0 and codes 0.
// packed != 0: codes in the packed pair/chunk layout; else row-major [N][K].
// byte of packed row R, weight e in the fp8 tile layout (described with kWfmtQ4)
__device__ __forceinline__ size_t f8_tile_offset(int R, int e, int nb) {
  const int rl = R % kQ4GroupRows, pair = rl >> 1, member = rl & 1;
  const int kb = e & 63, j = kb >> 4, kk = kb & 15, t = (kk & 7) >> 1, hi8 = kk >> 3, odd = kk & 1;
  const int lane = pair * 4 + t;
  return (static_cast<size_t>(R / kQ4GroupRows) * nb + (e >> 6)) * 1024 + (j >> 1) * 512 + lane * 16 + (j & 1) * 8 +
         4 * hi8 + 2 * member + odd;
}

__global__ void quant_pack_kernel(uint8_t* __restrict__ dst, float* __restrict__ scales,
                                  const __nv_bfloat16* __restrict__ s0, const __nv_bfloat16* __restrict__ s1,
                                  const __nv_bfloat16* __restrict__ s2, int mode, int N, int K, int CT, int nq,
                                  int nkv, int d, int layout) {
  constexpr int CH = 512;  // codes per row per chunk
  __shared__ float red[32];
  const int R = blockIdx.x, tid = threadIdx.x;
  const __nv_bfloat16* src = pack_src_row(s0, s1, s2, mode, R, N, K, nq, nkv, d);
  float amax = 0.f;
  if (src)
    for (int e = tid; e < K; e += blockDim.x) amax = fmaxf(amax, fabsf(__bfloat162float(src[e])));
  amax = warp_max(amax);
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  if (tid < 32) {
    float v = tid < static_cast<int>(blockDim.x >> 5) ? red[tid] : 0.f;
    v = warp_max(v);
    if (tid == 0) red[0] = v;
  }
  __syncthreads();
  const float scale = red[0] / 448.0f;
  if (tid == 0) scales[R] = scale;
  const int nb = (K + 63) / 64;  // tile units per tile
  const int n = layout == LAYOUT_PAIRS ? CT * CH : layout == LAYOUT_TILES ? nb * 64 : K;
  for (int e = tid; e < n; e += blockDim.x) {
    const float w = (src != nullptr && e < K) ? __bfloat162float(src[e]) : 0.f;
    const uint8_t code = scale > 0.f ? static_cast<uint8_t>(__nv_cvt_float_to_fp8(w / scale, __NV_SATFINITE, __NV_E4M3))
                                     : static_cast<uint8_t>(0);
    if (layout == LAYOUT_PAIRS) {
      const int c = e / CH, i = e - c * CH;
      dst[(static_cast<size_t>(R >> 1) * CT + c) * 2 * CH + (R & 1) * CH + i] = code;
    } else if (layout == LAYOUT_TILES) {
      dst[f8_tile_offset(R, e, nb)] = code;
    } else {
      dst[static_cast<size_t>(R) * K + e] = code;
    }
  }
}

// int4 block quantization (k2-burn README, "Quantization": int4 checkpoints
// with block size 64): one CTA of kQ4Chunk / 4 threads per (packed row R,
// chunk c); thread t takes weights 4t .. 4t + 3 of the chunk, 16 threads one
// 64-weight block.  s = max|w| / 7; code = w / s rounded to nearest, ties to
// even, clamped to [-7, 7]; a zero block gets s = 0 and codes 0.  Pairs:
// nibble c + 8, element 2i in the low nibble of byte i, into the int4 pair
// unit; tiles: nibble c + 8 OR-ed into the int4 tile unit (the rows of a tile
// word come from two CTAs, hence the atomic OR into a cleared buffer); plain:
// int8 codes [N][K], scales [N][ceil(K / 64)].  (Both unit layouts are
// described with kWfmtQ4.)
__global__ void __launch_bounds__(kQ4Chunk / 4) q4_pack_kernel(uint8_t* __restrict__ dst, float* __restrict__ scales,
                                                      const __nv_bfloat16* __restrict__ s0,
                                                      const __nv_bfloat16* __restrict__ s1,
                                                      const __nv_bfloat16* __restrict__ s2, int mode, int N, int K,
                                                      int CT, int nq, int nkv, int d, int layout) {
  const int R = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
  const __nv_bfloat16* src = pack_src_row(s0, s1, s2, mode, R, N, K, nq, nkv, d);
  const int e0 = c * kQ4Chunk + 4 * tid;  // the thread's first weight in the row
  float w[4];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[i] = (src != nullptr && e0 + i < K) ? __bfloat162float(src[e0 + i]) : 0.f;
    amax = fmaxf(amax, fabsf(w[i]));
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));  // the 16 threads
  const float s = __fdiv_rn(amax, 7.0f);
  int q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = s > 0.f ? max(-7, min(7, __float2int_rn(__fdiv_rn(w[i], s)))) : 0;
  const int blk = tid >> 4;  // the block within the chunk
  if (layout == LAYOUT_PAIRS) {
    uint8_t* unit = dst + (static_cast<size_t>(R >> 1) * CT + c) * kQ4Unit;
    const uint32_t b0 = static_cast<uint32_t>(q[0] + 8) | (static_cast<uint32_t>(q[1] + 8) << 4);
    const uint32_t b1 = static_cast<uint32_t>(q[2] + 8) | (static_cast<uint32_t>(q[3] + 8) << 4);
    *reinterpret_cast<uint16_t*>(unit + (R & 1) * (kQ4Chunk / 2) + 2 * tid) = static_cast<uint16_t>(b0 | (b1 << 8));
    if ((tid & 15) == 0)
      *reinterpret_cast<float*>(unit + kQ4Chunk + (R & 1) * (kQ4Chunk / kQ4Block) * 4 + blk * 4) = s;
  } else if (layout == LAYOUT_TILES) {
    const int nb = (K + kQ4Block - 1) / kQ4Block;  // blocks (units) per tile
    const int b = c * (kQ4Chunk / kQ4Block) + blk;
    if (b < nb) {
      const int rl = R % kQ4GroupRows, pair = rl >> 1, member = rl & 1;
      uint8_t* unit = dst + (static_cast<size_t>(R / kQ4GroupRows) * nb + b) * kQ4Unit;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int kb = 4 * (tid & 15) + i;  // position in the block
        const int j = kb >> 4, kk = kb & 15, t = (kk & 7) >> 1, hi8 = kk >> 3, odd = kk & 1;
        const int shift = 4 * member + 8 * hi8 + 16 * odd;
        atomicOr(reinterpret_cast<unsigned*>(unit + (pair * 4 + t) * 16 + j * 4),
                 static_cast<unsigned>(q[i] + 8) << shift);
      }
      if ((tid & 15) == 0) *reinterpret_cast<float*>(unit + 512 + pair * 8 + member * 4) = s;
    }
  } else if (R < N) {
    const int nb = (K + kQ4Block - 1) / kQ4Block;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (e0 + i < K) dst[static_cast<size_t>(R) * K + e0 + i] = static_cast<uint8_t>(static_cast<int8_t>(q[i]));
    const int b = c * (kQ4Chunk / kQ4Block) + blk;
    if ((tid & 15) == 0 && b < nb) scales[static_cast<size_t>(R) * nb + b] = s;
  }
}

template <typename WT>
cudaError_t launch_typed(const PackedGemvArgs& a, int epi, const cudaLaunchConfig_t& cfg) {
  switch (epi) {
    case EPI_STORE: return cudaLaunchKernelEx(&cfg, packed_gemv_kernel<WT, EPI_STORE>, a);
    case EPI_RESID: return cudaLaunchKernelEx(&cfg, packed_gemv_kernel<WT, EPI_RESID>, a);
    case EPI_QKV: return cudaLaunchKernelEx(&cfg, packed_gemv_kernel<WT, EPI_QKV>, a);
    case EPI_SWIGLU: return cudaLaunchKernelEx(&cfg, packed_gemv_kernel<WT, EPI_SWIGLU>, a);
    case EPI_ARGMAX: return cudaLaunchKernelEx(&cfg, packed_gemv_kernel<WT, EPI_ARGMAX>, a);
  }
  return cudaErrorInvalidValue;
}

template <typename WT>
cudaError_t set_attr(int bytes) {
  cudaError_t e;
  if ((e = set_kernel_smem(packed_gemv_kernel<WT, EPI_STORE>, bytes)))
    return e;
  if ((e = set_kernel_smem(packed_gemv_kernel<WT, EPI_RESID>, bytes)))
    return e;
  if ((e = set_kernel_smem(packed_gemv_kernel<WT, EPI_QKV>, bytes)))
    return e;
  if ((e = set_kernel_smem(packed_gemv_kernel<WT, EPI_SWIGLU>, bytes)))
    return e;
  return set_kernel_smem(packed_gemv_kernel<WT, EPI_ARGMAX>, bytes);
}

}  // namespace

size_t packed_bytes(int N, int K, int wbytes) {
  const int CH = 512 / wbytes;
  const size_t CT = (static_cast<size_t>(K) + CH - 1) / CH;
  const size_t npairs = (static_cast<size_t>(N) + 1) / 2;
  return npairs * CT * kUnitB;
}

int packed_grid(int N, int sms) {
  const int npairs = (N + 1) / 2;
  int g = sms < npairs ? sms : npairs;
  if (g > 1024) g = 1024;
  return g < 1 ? 1 : g;
}

bool packed_plan(PackedGemvArgs& a, int wbytes, size_t smem_budget, int max_slots) {
  if (wbytes != 2 && wbytes != 4) return false;
  const int EPL = 16 / wbytes;
  const int CH = 32 * EPL;
  if (a.N <= 0 || a.K <= 0 || a.K % 4) return false;
  if (a.gain && (a.groups < 1 || a.groups > 4 || a.K % a.groups || (a.K / a.groups) % 4)) return false;
  a.CT = (a.K + CH - 1) / CH;
  a.x_bytes = static_cast<uint32_t>(a.CT) * CH * 4;
  if (a.x_bytes >= smem_budget) return false;
  const size_t ring = smem_budget - a.x_bytes;
  // the largest copies (up to 5 KB) that still leave two slots per warp
  for (int su = 5; su >= 1; --su) {
    const size_t ns = ring / (static_cast<size_t>(kPackedWarps) * su * kUnitB);
    if (ns >= 2) {
      a.SU = su;
      a.NS = static_cast<int>(ns > static_cast<size_t>(max_slots) ? max_slots : ns);
      return true;
    }
  }
  return false;
}

size_t packed_smem_bytes(const PackedGemvArgs& a) {
  return static_cast<size_t>(kPackedWarps) * a.NS * a.SU * kUnitB + a.x_bytes;
}

cudaError_t packed_init_attrs() {
  cudaError_t e = set_attr<__nv_bfloat16>(200 * 1024);
  if (e != cudaSuccess) return e;
  return set_attr<float>(200 * 1024);
}

cudaError_t launch_packed_gemv(const PackedGemvArgs& a, int wbytes, int epi, int grid, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPackedThreads);
  cfg.dynamicSmemBytes = packed_smem_bytes(a);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return wbytes == 2 ? launch_typed<__nv_bfloat16>(a, epi, cfg) : launch_typed<float>(a, epi, cfg);
}

cudaError_t launch_pack(void* dst, const void* src0, const void* src1, const void* src2, int mode, int N, int K,
                        int wbytes, int nq, int nkv, int d, cudaStream_t s) {
  const int CH = 512 / wbytes;
  const int CT = (K + CH - 1) / CH;
  const int rows = 2 * ((N + 1) / 2);
  if (wbytes == 2)
    pack_kernel<__nv_bfloat16><<<rows, 256, 0, s>>>(
        static_cast<__nv_bfloat16*>(dst), static_cast<const __nv_bfloat16*>(src0),
        static_cast<const __nv_bfloat16*>(src1), static_cast<const __nv_bfloat16*>(src2), mode, N, K, CT, nq, nkv, d);
  else
    pack_kernel<float><<<rows, 256, 0, s>>>(static_cast<float*>(dst), static_cast<const float*>(src0),
                                            static_cast<const float*>(src1), static_cast<const float*>(src2), mode, N,
                                            K, CT, nq, nkv, d);
  return cudaGetLastError();
}

// One CTA of 256 threads per (packed row R, bf16 chunk c): weight k = 256 c + t.
__global__ void __launch_bounds__(256) f8_expand_kernel(__nv_bfloat16* __restrict__ dst,
                                                        const uint8_t* __restrict__ src, int CT8, int CT16, int nb) {
  const int R = blockIdx.x, c = blockIdx.y, k = c * 256 + threadIdx.x;
  const int c8 = k >> 9, i8 = k & 511;
  // nb > 0: the source is in tile units (nb per tile); weights past the tile's
  // blocks are zero
  const uint8_t code = nb > 0 ? ((k >> 6) < nb ? src[f8_tile_offset(R, k, nb)] : static_cast<uint8_t>(0))
                              : src[(static_cast<size_t>(R >> 1) * CT8 + c8) * 1024 + (R & 1) * 512 + i8];
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);
  dst[(static_cast<size_t>(R >> 1) * CT16 + c) * 512 + (R & 1) * 256 + threadIdx.x] =
      __float2bfloat16_rn(__half2float(__half(h)));
}

cudaError_t launch_f8_expand(void* dst, const uint8_t* src, int N, int K, bool tiles, cudaStream_t s) {
  const int CT8 = (K + 511) / 512, CT16 = (K + 255) / 256, rows = 2 * ((N + 1) / 2);
  if (rows <= 0 || CT16 <= 0) return cudaSuccess;
  f8_expand_kernel<<<dim3(rows, CT16), 256, 0, s>>>(static_cast<__nv_bfloat16*>(dst), src, CT8, CT16,
                                                    tiles ? (K + 63) / 64 : 0);
  return cudaGetLastError();
}

// The int4 weights of a packed matrix (pair or tile units) dequantized for
// the tensor-core prefill: w = code * scale (fp32, as the decode step scales
// each block), split into bf16 halves w_hi = bf16(w), w_lo = bf16(w - w_hi), in
// the bf16 packed layout (pairs of rows in 256-weight chunks).  One CTA of 256
// threads per (packed row R, bf16 chunk c): weight k = 256 c + t.
__global__ void __launch_bounds__(256) q4_dequant_kernel(__nv_bfloat16* __restrict__ hi, __nv_bfloat16* __restrict__ lo,
                                                         const uint8_t* __restrict__ src, int K, int CT16, int tiles) {
  const int R = blockIdx.x, c = blockIdx.y, k = c * 256 + threadIdx.x;
  float w = 0.f;
  if (k < K) {
    if (tiles) {
      const int nb = (K + kQ4Block - 1) / kQ4Block;
      const int rl = R % kQ4GroupRows, pair = rl >> 1, member = rl & 1;
      const int kb = k & 63, j = kb >> 4, kk = kb & 15, t = (kk & 7) >> 1, hi8 = kk >> 3, odd = kk & 1;
      const uint8_t* unit = src + (static_cast<size_t>(R / kQ4GroupRows) * nb + (k >> 6)) * kQ4Unit;
      const uint32_t word = *reinterpret_cast<const uint32_t*>(unit + (pair * 4 + t) * 16 + j * 4);
      const int code = static_cast<int>((word >> (4 * member + 8 * hi8 + 16 * odd)) & 15u) - 8;
      w = static_cast<float>(code) * *reinterpret_cast<const float*>(unit + 512 + pair * 8 + member * 4);
    } else {
      const int CT = (K + kQ4Chunk - 1) / kQ4Chunk, i = k % kQ4Chunk;
      const uint8_t* unit = src + (static_cast<size_t>(R >> 1) * CT + k / kQ4Chunk) * kQ4Unit;
      const uint8_t b = unit[(R & 1) * (kQ4Chunk / 2) + (i >> 1)];
      const int code = static_cast<int>((i & 1) ? (b >> 4) : (b & 15u)) - 8;
      w = static_cast<float>(code) *
          *reinterpret_cast<const float*>(unit + kQ4Chunk + (R & 1) * (kQ4Chunk / kQ4Block) * 4 + (i / kQ4Block) * 4);
    }
  }
  const __nv_bfloat16 h = __float2bfloat16_rn(w);
  const size_t o = (static_cast<size_t>(R >> 1) * CT16 + c) * 512 + (R & 1) * 256 + threadIdx.x;
  hi[o] = h;
  lo[o] = __float2bfloat16_rn(w - __bfloat162float(h));
}

cudaError_t launch_q4_dequant(void* hi, void* lo, const uint8_t* src, int N, int K, bool tiles, cudaStream_t s) {
  const int CT16 = (K + 255) / 256, rows = 2 * ((N + 1) / 2);
  if (rows <= 0 || CT16 <= 0) return cudaSuccess;
  q4_dequant_kernel<<<dim3(rows, CT16), 256, 0, s>>>(static_cast<__nv_bfloat16*>(hi), static_cast<__nv_bfloat16*>(lo),
                                                     src, K, CT16, tiles ? 1 : 0);
  return cudaGetLastError();
}

size_t f8_packed_bytes(int N, int K, bool tiles) {
  if (!tiles) return packed_bytes(N, K, 1);
  return (static_cast<size_t>(N) + kQ4GroupRows - 1) / kQ4GroupRows * ((static_cast<size_t>(K) + 63) / 64) * 1024;
}

size_t q4_packed_bytes(int N, int K, bool tiles) {
  if (!tiles) {
    const size_t CT = (static_cast<size_t>(K) + kQ4Chunk - 1) / kQ4Chunk;
    return (static_cast<size_t>(N) + 1) / 2 * CT * kQ4Unit;
  }
  const size_t nb = (static_cast<size_t>(K) + kQ4Block - 1) / kQ4Block;
  const size_t groups = (static_cast<size_t>(N) + kQ4GroupRows - 1) / kQ4GroupRows;
  return groups * nb * kQ4Unit;
}

cudaError_t launch_q4_pack(uint8_t* dst, float* scales, const void* src0, const void* src1, const void* src2,
                           int mode, int N, int K, int nq, int nkv, int d, int layout, cudaStream_t s) {
  const int CT = (K + kQ4Chunk - 1) / kQ4Chunk;
  const int rows = layout == LAYOUT_TILES   ? kQ4GroupRows * ((N + kQ4GroupRows - 1) / kQ4GroupRows)
                   : layout == LAYOUT_PAIRS ? 2 * ((N + 1) / 2)
                                        : N;
  if (rows <= 0 || CT <= 0) return cudaSuccess;
  if (layout == LAYOUT_TILES) {
    const cudaError_t e = cudaMemsetAsync(dst, 0, q4_packed_bytes(N, K, true), s);
    if (e != cudaSuccess) return e;
  }
  q4_pack_kernel<<<dim3(rows, CT), kQ4Chunk / 4, 0, s>>>(dst, scales, static_cast<const __nv_bfloat16*>(src0),
                                                static_cast<const __nv_bfloat16*>(src1),
                                                static_cast<const __nv_bfloat16*>(src2), mode, N, K, CT, nq, nkv, d,
                                                layout);
  return cudaGetLastError();
}

cudaError_t launch_quant_pack(uint8_t* dst, float* scales, const void* src0, const void* src1, const void* src2,
                              int mode, int N, int K, int nq, int nkv, int d, int layout, cudaStream_t s) {
  const int CT = (K + 511) / 512;
  const int rows = layout == LAYOUT_TILES   ? kQ4GroupRows * ((N + kQ4GroupRows - 1) / kQ4GroupRows)
                   : layout == LAYOUT_PAIRS ? 2 * ((N + 1) / 2)
                                            : N;
  if (rows <= 0) return cudaSuccess;
  quant_pack_kernel<<<rows, 256, 0, s>>>(dst, scales, static_cast<const __nv_bfloat16*>(src0),
                                         static_cast<const __nv_bfloat16*>(src1),
                                         static_cast<const __nv_bfloat16*>(src2), mode, N, K, CT, nq, nkv, d,
                                         layout);
  return cudaGetLastError();
}

}  // namespace k2
