// Token sampling from logits (k2-burn README, "Sampling + greedy
// generation": temperature / top-k / top-p / min-p / repetition penalty with
// a seeded RNG; temperature 0 stays the greedy argmax of the decode step).
//
// One cooperative launch: `cpr` CTAs per row, each owning a 32-aligned slice
// of the vocabulary.  Exact filters over the whole vocabulary, done as radix
// selections whose histograms are merged in global memory with integer
// atomics (so the order of the merges does not matter), separated by a
// bounded grid barrier:
//   1. repetition penalty: the row's seen token ids set bits of a bitmap;
//      l -> l / r for l > 0, l * r otherwise, once per distinct id;
//   2. z = l / T and its maximum;
//   3. top-k: the k-th largest z (three 11/11/10-bit digit passes); kept: z >= it;
//   4. weights w = exp(z - zmax) in [0, 1] (own exp, see exp_neg), integer
//      masses m = floor(w * 2^32), their total W over the top-k survivors;
//   5. top-p: the smallest weight key whose strictly-heavier mass is below
//      top_p * W (three passes over the bits of w); kept: w >= it, so tied
//      weights are kept or dropped together;
//   6. min-p: kept: w >= min_p (w is the probability relative to the maximum);
//   7. one Philox4x32-10 draw u (counter = the position the token takes, the
//      sequence; key = the seed) picks the first index, in vocabulary order,
//      whose inclusive prefix of kept masses exceeds floor(u * total).
// Every decision is made on integers or on IEEE-rounded fp32 operations (no
// contraction), so a plain implementation of the same definitions reproduces
// the token bit for bit.
#include <math.h>

#include "k2_kernels.h"
#include "k2_common.cuh"

namespace k2 {

namespace {

constexpr int ST = kSampleThreads;
constexpr int NB = kSampleBins;  // 2048 = 11-bit digits
typedef unsigned long long u64;

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011): ten rounds of two 32x32->64 multiplications,
// the key bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const u64 p0 = static_cast<u64>(0xD2511F53u) * c.x;
    const u64 p1 = static_cast<u64>(0xCD9E8D57u) * c.z;
    c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ k0, static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ c.w ^ k1, static_cast<uint32_t>(p0));
  }
  return c;
}

// exp(x) for x <= 0 in fp32 from IEEE-rounded multiplies and adds only:
// Cody-Waite reduction x = n ln2 + r (ln2 split into a 12-bit head and a
// tail), the degree-7 Taylor polynomial of exp(r) for |r| <= ln2 / 2 in
// Horner form, then the exact scaling by 2^n.  Zero below -87 (under 2^-125,
// a mass of 0 at 2^32 resolution).
__device__ __forceinline__ float exp_neg(float x) {
  if (!(x > -87.0f)) return 0.f;
  const float n = rintf(__fmul_rn(x, 1.44269504088896341f));
  float r = __fsub_rn(x, __fmul_rn(n, 0.693145751953125f));
  r = __fsub_rn(r, __fmul_rn(n, 1.42860676533018708e-06f));
  float p = 1.98412698412698413e-4f;                   // 1/7!
  p = __fadd_rn(__fmul_rn(p, r), 1.38888888888888889e-3f);  // 1/6!
  p = __fadd_rn(__fmul_rn(p, r), 8.33333333333333333e-3f);  // 1/5!
  p = __fadd_rn(__fmul_rn(p, r), 4.16666666666666667e-2f);  // 1/4!
  p = __fadd_rn(__fmul_rn(p, r), 1.66666666666666667e-1f);  // 1/3!
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  return __fmul_rn(p, __int_as_float((static_cast<int>(n) + 127) << 23));
}

// order-preserving unsigned key of a float (NaN never reaches it)
__device__ __forceinline__ uint32_t okey(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float okey_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ u64 wmass(float w) { return static_cast<u64>(w * 4294967296.0f); }

// the three digits of a 32-bit key: bits 21..31, 10..20, 0..9
__device__ __forceinline__ int dshift(int p) { return p == 0 ? 21 : p == 1 ? 10 : 0; }
__device__ __forceinline__ uint32_t dmask(int p) { return p == 2 ? 0x3ffu : 0x7ffu; }

struct RowScratch {
  unsigned* zmax;
  u64* wsum;
  u64* part;
  unsigned* cnt;  // [3][NB]
  u64* mass;      // [3][NB]
  unsigned* bitmap;
};

__device__ __forceinline__ RowScratch row_scratch(const SampleArgs& a, int row) {
  uint8_t* base = a.scratch + kSampleBarBytes + static_cast<size_t>(row) * a.row_bytes;
  RowScratch s;
  s.zmax = reinterpret_cast<unsigned*>(base);
  s.wsum = reinterpret_cast<u64*>(base + 8);
  s.part = reinterpret_cast<u64*>(base + 16);
  s.cnt = reinterpret_cast<unsigned*>(base + 16 + 8 * kSampleCtaMax);
  s.mass = reinterpret_cast<u64*>(base + 16 + 8 * kSampleCtaMax + 4 * 3 * NB);
  s.bitmap = reinterpret_cast<unsigned*>(base + 16 + 8 * kSampleCtaMax + 12 * 3 * NB);
  return s;
}

// Grid barrier number `n` (1, 2, ...): every CTA arrives once per barrier.
// The counter was zeroed before the launch; the wait is bounded.
__device__ bool grid_barrier(unsigned* bar, unsigned n, unsigned G, unsigned* guard) {
  __shared__ int ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    ok = 1;
    __threadfence();
    atomicAdd(bar, 1u);
    const uint64_t t0 = globaltimer();
    while (true) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
      if (v >= n * G) break;
      if (globaltimer() - t0 > kWaitLimitNs) {
        atomicOr(guard, GUARD_TIMEOUT);
        ok = 0;
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();
  return ok != 0;
}

// Warp 0 finds the digit: from the highest bin down, the first at which the
// running value (plus `above`) satisfies `reached`; *above_out = the value of
// the bins above it.  Three levels (groups of bins, sub-groups, bins), each a
// suffix scan over the lanes; every CTA runs it on the same merged bins.
template <typename T, typename Reached>
__device__ int pick_digit(const T* bins, int nbins, T above, Reached reached, T* above_out) {
  __shared__ int dsel;
  __shared__ T asel;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int lo = 0, n = nbins;
    T acc = above;
    int d = 0;
    bool found = false;
    while (true) {
      const int q = n > 32 ? n / 32 : 1;  // bins per lane at this level
      T own = 0;
      if (n > 32) {
        for (int b = 0; b < q; ++b) own += bins[lo + lane * q + (b + lane) % q];  // rotated: no bank conflicts
      } else if (lane < n) {
        own = bins[lo + lane];
      }
      T suf = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const T v = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += v;
      }
      const T excl = suf - own;  // the bins of higher lanes
      const unsigned m = __ballot_sync(0xffffffffu, reached(acc + suf) && !reached(acc + excl));
      if (m == 0) break;  // nothing reaches (not for consistent bins)
      const int hl = 31 - __clz(m);
      acc += __shfl_sync(0xffffffffu, excl, hl);
      lo += hl * q;
      if (q == 1) {
        d = lo;
        found = true;
        break;
      }
      n = q;
    }
    if (!found) {  // the lowest bin, keeping everything
      d = 0;
      acc = above;
      for (int b = 1; b < nbins; ++b) acc += bins[b];
    }
    if (lane == 0) {
      dsel = d;
      asel = acc;
    }
  }
  __syncthreads();
  *above_out = asel;
  return dsel;
}

__global__ void __launch_bounds__(ST) sample_kernel(const SampleArgs a) {
  extern __shared__ float zs[];  // z of this CTA's slice of the vocabulary
  __shared__ unsigned hc[NB];    // this CTA's histogram, then the merged one
  __shared__ u64 hm[NB];
  __shared__ float redf[ST / 32];
  __shared__ u64 redu[ST / 32];
  __shared__ u64 scan_tot[ST / 32];
  __shared__ int found;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cpr = a.ctas_per_row;
  const int row = blockIdx.x / cpr, j = blockIdx.x - (blockIdx.x / cpr) * cpr;
  const unsigned G = gridDim.x;
  const int V = a.vocab;
  const float* lg = a.logits + static_cast<size_t>(row) * a.ld;
  const RowScratch rs = row_scratch(a, row);
  unsigned* bar = reinterpret_cast<unsigned*>(a.scratch);
  const int s0 = static_cast<int>((static_cast<long long>(V) * j / cpr) & ~31LL);
  const int s1 = j == cpr - 1 ? V : static_cast<int>((static_cast<long long>(V) * (j + 1) / cpr) & ~31LL);
  const int ns = s1 - s0;
  unsigned nbar = 0;
  const bool pen = a.seen != nullptr && a.penalty != 1.0f;
  const bool topk = a.top_k > 0 && a.top_k < V;
  const bool topp = a.top_p < 1.0f;

  // merged bins of pass p into shared memory, after the barrier
  auto merge_counts = [&](int p) -> bool {
    unsigned* gc = rs.cnt + p * NB;
    for (int b = tid; b < NB; b += ST)
      if (hc[b]) atomicAdd(gc + b, hc[b]);
    if (!grid_barrier(bar, ++nbar, G, a.guard)) return false;
    for (int b = tid; b < NB; b += ST) hc[b] = __ldcg(gc + b);
    __syncthreads();
    return true;
  };
  auto merge_masses = [&](int p) -> bool {
    u64* gm = rs.mass + p * NB;
    for (int b = tid; b < NB; b += ST)
      if (hm[b]) atomicAdd(gm + b, hm[b]);
    if (!grid_barrier(bar, ++nbar, G, a.guard)) return false;
    for (int b = tid; b < NB; b += ST) hm[b] = __ldcg(gm + b);
    __syncthreads();
    return true;
  };
  auto clear_bins = [&]() {
    for (int b = tid; b < NB; b += ST) {
      hc[b] = 0;
      hm[b] = 0;
    }
    __syncthreads();
  };

  // 1. the row's seen ids
  if (pen) {
    const int n = a.seen_len[row];
    const int* sp = a.seen + static_cast<size_t>(row) * a.seen_stride;
    for (int i = j * ST + tid; i < n; i += cpr * ST) {
      const int id = sp[i];
      if (id >= 0 && id < V) atomicOr(&rs.bitmap[id >> 5], 1u << (id & 31));
    }
    if (!grid_barrier(bar, ++nbar, G, a.guard)) return;
  }

  // 2. z of the slice (kept in shared memory), its maximum, and the first
  // top-k histogram (digit 0 of the order key)
  clear_bins();
  {
    float mz = -INFINITY;
    for (int t = tid; t < ns; t += ST) {
      const int i = s0 + t;
      float l = __ldcg(lg + i);
      float z;
      if (!(l == l)) {
        z = -INFINITY;
      } else {
        if (pen && ((__ldcg(rs.bitmap + (i >> 5)) >> (i & 31)) & 1u)) l = l > 0.f ? l / a.penalty : l * a.penalty;
        z = l / a.temperature;
      }
      zs[t] = z;
      mz = fmaxf(mz, z);
      if (topk) atomicAdd(&hc[(okey(z) >> dshift(0)) & dmask(0)], 1u);
    }
    mz = warp_max(mz);
    if (lane == 0) redf[warp] = mz;
    __syncthreads();
    if (tid == 0) {
      float t = redf[0];
      for (int w = 1; w < ST / 32; ++w) t = fmaxf(t, redf[w]);
      atomicMax(rs.zmax, okey(t));
    }
  }
  if (topk) {
    if (!merge_counts(0)) return;
  } else if (!grid_barrier(bar, ++nbar, G, a.guard)) {
    return;
  }
  const float zmax = okey_inv(__ldcg(rs.zmax));

  // 3. top-k: the key of the k-th largest z
  uint32_t kkey = 0;
  if (topk) {
    uint32_t prefix = 0, mask = 0;
    unsigned need = static_cast<unsigned>(a.top_k);
    for (int p = 0; p < 3; ++p) {
      if (p > 0) {
        clear_bins();
        for (int t = tid; t < ns; t += ST) {
          const uint32_t k = okey(zs[t]);
          if ((k & mask) == prefix) atomicAdd(&hc[(k >> dshift(p)) & dmask(p)], 1u);
        }
        __syncthreads();
        if (!merge_counts(p)) return;
      }
      unsigned above = 0;
      const int d = pick_digit<unsigned>(hc, static_cast<int>(dmask(p)) + 1, 0u,
                                         [&](unsigned v) { return v >= need; }, &above);
      need -= above;
      prefix |= static_cast<uint32_t>(d) << dshift(p);
      mask |= dmask(p) << dshift(p);
    }
    kkey = prefix;
  }

  // 4./5. top-p over the weights of the top-k survivors; the first pass's
  // merged bins also give their total W
  uint32_t pkey = 0;
  if (topp) {
    uint32_t prefix = 0, mask = 0;
    u64 above = 0;
    double target = 0.0;
    for (int p = 0; p < 3; ++p) {
      clear_bins();
      for (int t = tid; t < ns; t += ST) {
        const float z = zs[t];
        if (okey(z) < kkey) continue;
        const float w = exp_neg(z - zmax);
        const uint32_t k = __float_as_uint(w);
        if ((k & mask) == prefix) atomicAdd(&hm[(k >> dshift(p)) & dmask(p)], wmass(w));
      }
      __syncthreads();
      if (!merge_masses(p)) return;
      if (p == 0) {
        u64 t = 0;
        for (int b = tid; b < NB; b += ST) t += hm[b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) redu[warp] = t;
        __syncthreads();
        u64 W = 0;
        for (int w = 0; w < ST / 32; ++w) W += redu[w];
        target = static_cast<double>(a.top_p) * static_cast<double>(W);
        __syncthreads();
      }
      const int d = pick_digit<u64>(hm, static_cast<int>(dmask(p)) + 1, above,
                                    [&](u64 v) { return static_cast<double>(v) >= target; }, &above);
      prefix |= static_cast<uint32_t>(d) << dshift(p);
      mask |= dmask(p) << dshift(p);
    }
    pkey = prefix;
  }

  // 6./7. the kept masses of this slice, then the draw
  auto kept_mass = [&](int t) -> u64 {
    const float z = zs[t];
    if (okey(z) < kkey) return 0;
    const float w = exp_neg(z - zmax);
    if (__float_as_uint(w) < pkey || w < a.min_p) return 0;
    return wmass(w);
  };
  {
    u64 acc = 0;
    for (int t = tid; t < ns; t += ST) acc += kept_mass(t);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) redu[warp] = acc;
    __syncthreads();
    if (tid == 0) {
      u64 t = 0;
      for (int w = 0; w < ST / 32; ++w) t += redu[w];
      rs.part[j] = t;
    }
    if (!grid_barrier(bar, ++nbar, G, a.guard)) return;
  }
  // every CTA of the row: the total, the draw, the CTA whose slice holds it
  u64 total = 0, base = 0, target = 0;
  int owner = -1;
  {
    for (int c = 0; c < cpr; ++c) total += __ldcg(rs.part + c);
    const uint4 x = philox4x32_10(make_uint4(static_cast<uint32_t>(a.counter[row]),
                                             static_cast<uint32_t>(a.first_seq + row), 0u, 0u),
                                  a.key0, a.key1);
    const u64 r = x.x >> 8;  // 24 random bits: u = r / 2^24
    target = (total >> 24) * r + (((total & 0xFFFFFFull) * r) >> 24);  // floor(u * total) < total
    u64 run = 0;
    for (int c = 0; c < cpr; ++c) {
      const u64 v = __ldcg(rs.part + c);
      if (owner < 0 && run + v > target) {
        owner = c;
        base = run;
      }
      run += v;
    }
  }
  if (owner < 0) {  // no kept mass at all (every logit NaN or -inf)
    if (j == 0 && tid == 0) {
      atomicOr(a.guard, GUARD_NAN);
      a.next[row] = 0;
    }
    return;
  }
  if (owner != j) return;
  // each thread a contiguous run of the slice: one block scan of the runs'
  // masses, then the thread whose run holds the target walks it
  {
    const int per = (ns + ST - 1) / ST;
    const int t0 = tid * per, t1 = min(ns, t0 + per);
    u64 own = 0;
    for (int t = t0; t < t1; ++t) own += kept_mass(t);
    u64 inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const u64 v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane == 31) scan_tot[warp] = inc;
    if (tid == 0) found = -1;
    __syncthreads();
    u64 run = base + inc - own;
    for (int w = 0; w < warp; ++w) run += scan_tot[w];
    if (own > 0 && run <= target && target < run + own) {  // exactly one thread
      for (int t = t0; t < t1; ++t) {
        run += kept_mass(t);
        if (run > target) {
          found = s0 + t;
          break;
        }
      }
    }
    __syncthreads();
  }
  if (tid == 0) {
    if (found < 0) {
      atomicOr(a.guard, GUARD_NAN);
      found = 0;
    }
    a.next[row] = found;
  }
}

}  // namespace

// dynamic shared memory of one CTA: z of its slice (32-aligned bounds)
size_t sample_smem_bytes(int vocab, int cpr) {
  return 4 * (static_cast<size_t>((vocab + cpr - 1) / cpr) + 64);
}

int sample_ctas_per_row(int rows, int vocab) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSampleSmemMax) != cudaSuccess)
    return 0;
  for (int cpr = kSampleCtaMax; cpr >= 1; --cpr) {
    const size_t smem = sample_smem_bytes(vocab, cpr);
    if (smem > static_cast<size_t>(kSampleSmemMax)) break;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sample_kernel, ST, smem) != cudaSuccess) return 0;
    if (per_sm >= 1 && static_cast<long long>(rows) * cpr <= static_cast<long long>(sms) * per_sm) return cpr;
  }
  return 0;
}

size_t sample_row_bytes(int vocab) {
  const size_t b = 16 + 8 * static_cast<size_t>(kSampleCtaMax) + 12 * 3 * static_cast<size_t>(NB) +
                   4 * ((static_cast<size_t>(vocab) + 31) / 32);
  return (b + 255) / 256 * 256;
}

cudaError_t launch_sample(const SampleArgs& a, int rows, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(a.scratch, 0, kSampleBarBytes + static_cast<size_t>(rows) * a.row_bytes, s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows * a.ctas_per_row);
  cfg.blockDim = dim3(ST);
  cfg.dynamicSmemBytes = sample_smem_bytes(a.vocab, a.ctas_per_row);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<SampleArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(sample_kernel), args);
}

namespace {
// Philox4x32-10 outputs for counters (c, 0, 0, 0), c = first .. first + n - 1,
// under key (k0, k1): out[4 * i + w] (the generator of the sampler, exposed
// for its known-answer and cross-implementation checks).
__global__ void philox_kernel(uint32_t first, int n, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1,
                              uint32_t* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint4 x = philox4x32_10(make_uint4(first + static_cast<uint32_t>(i), c1, c2, c3), k0, k1);
  out[4 * i] = x.x;
  out[4 * i + 1] = x.y;
  out[4 * i + 2] = x.z;
  out[4 * i + 3] = x.w;
}

}  // namespace

cudaError_t launch_philox(uint32_t first, int n, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1,
                          uint32_t* out, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  philox_kernel<<<(n + 255) / 256, 256, 0, s>>>(first, n, c1, c2, c3, k0, k1, out);
  return cudaGetLastError();
}

}  // namespace k2
