// Persistent decode-step kernel: one cooperative launch runs a whole batch-1
// token (embedding row, every decoder layer, final norm, lm_head, argmax) on
// exactly one CTA per SM.
//
// Why one kernel: at batch 1 every step of the layer (k2-burn README,
// "Project layout": norm+attn residual, norm+mlp residual) is a short,
// HBM-bound pass (5 to 105 MB).  As separate launches they lose much of
// their time to ramp-up and tails, and under programmatic dependent launch
// the CTAs of a new kernel land on whatever SMs have room (measured: GEMV
// CTAs doubled up on 64-74 SMs while others idled).  Here every phase uses
// all SMs once and phases are separated by a grid barrier.
//
// The weights and cached K/V rows never depend on the activations, so each
// warp streams them continuously: its producer lane walks one fixed sequence
// of 10 KB slots spanning every phase of the step (its share of the QKV
// weights, then its K/V tiles, then its o_proj, gate/up, down weights, then
// the next layer's ...) and refills a ring slot as soon as it is consumed.
// The next phase's data is therefore already in flight while the CTAs meet
// at a barrier and rebuild the input vector.  Each refill is one bulk TMA
// copy (cp.async.bulk, mbarrier complete_tx) of a contiguous run of the
// packed weights (pairs of rows in 512-byte chunks) or of one 16-key K/V
// tile; a probe on this GPU streamed 6.9-7.4 TB/s with this consumer and
// 5-10 KB copies.
//
// Phases of a layer: QKV GEMV (+ GroupedRMSNorm, + split-half RoPE) | GQA
// attention partials per (KV head, key split) with the KV append | split merge
// | o_proj GEMV + residual | gate/up GEMV + SwiGLU | down GEMV + residual.
// Then final norm + lm_head GEMV + first-index argmax (kimi-k3-in-c k3_run.c,
// `argmax_`).
//
// Memory model: a phase's outputs are written with ordinary stores; the grid
// barrier (CTA barrier, gpu-scope fence, release add, acquire poll) orders
// them before every read in later phases, and those reads go to L2 (ld.cg or
// TMA), never to a possibly stale L1 line.  Every wait is bounded.
#include <math.h>

#include <type_traits>

#include "k2_kernels.h"
#include "k2_common.cuh"

namespace k2 {

namespace {

constexpr int MT = kMegaThreads;
constexpr int MW = MT / 32;
constexpr int NS = kMegaSlots;
constexpr int SB = kMegaSlotBytes;
constexpr int kUnit = 1024;      // one packed unit: a 512-byte chunk of both rows of a pair
constexpr int SU = SB / kUnit;   // packed units per slot
// keys per attention tile: the K and V rows (plus int8 scales) fit one slot
template <int D, typename KVT>
constexpr int tile_keys() {
  return (2 * kMegaTK * D * static_cast<int>(sizeof(KVT)) + 4 * kMegaTK <= SB) ? kMegaTK
         : (2 * (kMegaTK / 2) * D * static_cast<int>(sizeof(KVT)) + 4 * (kMegaTK / 2) <= SB) ? kMegaTK / 2
                                                                                               : 0;
}
constexpr int kPhases = 6;       // per layer: QKV, ATTN, MERGE, O, GU, DOWN
enum { PH_QKV = 0, PH_ATTN = 1, PH_MERGE = 2, PH_O = 3, PH_GU = 4, PH_DOWN = 5 };

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

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add_u32(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct MegaShared {
  uint64_t full[MW][NS];
  float ss[MW][4];
  float rs[4];
  int rec_pair[MW][2];
  float rec_val[MW][2][2];
  int rec_n[MW];
  Best best[MW];
  int flag;
  int ok;
  float rsd[2 * kMegaPairsMax];     // residual rows of this CTA (RESID phases)
  float2 rope[kMegaPairsMax];       // (cos, sin) of this CTA's pairs (QKV phase)
  float newkv[2][128];              // the new token's K and V rows (attention, head_dim <= 128)
};

// Grid barrier number bi of this launch: every CTA adds one to the arrival
// counter and waits until it reaches (bi + 1) * gridDim.x.  The counter is
// set back to 0 by the last CTA of the launch.  False if the wait ran out.
__device__ bool grid_sync(const MegaArgs& a, MegaShared& sh, int bi) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned target = static_cast<unsigned>(bi + 1) * gridDim.x;
    __threadfence();
    red_release_add_u32(a.bar_count, 1u);
    int ok = 1;
    if (ld_acquire_u32(a.bar_count) < target) {
      const uint64_t t0 = globaltimer();
      while (ld_acquire_u32(a.bar_count) < target) {
        if (globaltimer() - t0 > kWaitLimitNs) {
          atomicOr(a.guard, GUARD_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    sh.ok = ok;
  }
  __syncthreads();
  return sh.ok != 0;
}

// ---- static description of the step ------------------------------------------------
struct GDesc {
  const uint8_t* W;
  int N, K, CT;
  const void* gain;
};

__device__ __forceinline__ GDesc gdesc(const MegaArgs& a, int q, int qkv_n, int head_dim) {
  GDesc d;
  const int l = q / kPhases, j = q - (q / kPhases) * kPhases;
  if (l >= a.n_layers) {  // the lm_head phase
    d.W = static_cast<const uint8_t*>(a.lm_head);
    d.N = a.vocab;
    d.K = a.hidden;
    d.CT = a.g_lm.CT;
    d.gain = a.final_norm;
    return d;
  }
  const LayerPtrs& lp = a.layers[l];
  if (j == PH_QKV) {
    d.W = static_cast<const uint8_t*>(lp.wqkv); d.N = qkv_n; d.K = a.hidden; d.CT = a.g_qkv.CT; d.gain = lp.attn_norm;
  } else if (j == PH_O) {
    d.W = static_cast<const uint8_t*>(lp.wo); d.N = a.hidden; d.K = a.nq * head_dim; d.CT = a.g_o.CT; d.gain = nullptr;
  } else if (j == PH_GU) {
    d.W = static_cast<const uint8_t*>(lp.wgu); d.N = 2 * a.inter; d.K = a.hidden; d.CT = a.g_gu.CT; d.gain = lp.mlp_norm;
  } else {
    d.W = static_cast<const uint8_t*>(lp.wdown); d.N = a.hidden; d.K = a.inter; d.CT = a.g_down.CT; d.gain = nullptr;
  }
  return d;
}

struct GRange {
  int p0, p1, ua, ub, nslots;  // the CTA's pairs [p0, p1); the warp's units [ua, ub)
};

__device__ __forceinline__ GRange g_range(const GDesc& d, int cta, int G, int warp) {
  const int npairs = (d.N + 1) / 2;
  GRange r;
  r.p0 = static_cast<int>((static_cast<long long>(npairs) * cta) / G);
  r.p1 = static_cast<int>((static_cast<long long>(npairs) * (cta + 1)) / G);
  const long long U = static_cast<long long>(r.p1 - r.p0) * d.CT;
  r.ua = static_cast<int>((U * warp) / MW);
  r.ub = static_cast<int>((U * (warp + 1)) / MW);
  r.nslots = (r.ub - r.ua + SU - 1) / SU;
  return r;
}

struct AItem {
  int g, sp, k0, k1, ntile;
};

template <int TKM>
__device__ __forceinline__ AItem a_item(const MegaArgs& a, int item, int L) {
  AItem it;
  it.g = item / a.nsplit;
  it.sp = item - it.g * a.nsplit;
  const int ns = a.nsplit;
  it.k0 = min(L, static_cast<int>((static_cast<long long>(L) * it.sp) / ns) & ~7);
  it.k1 = (it.sp == ns - 1) ? L : min(L, static_cast<int>((static_cast<long long>(L) * (it.sp + 1)) / ns) & ~7);
  it.ntile = it.k1 > it.k0 ? (it.k1 - it.k0 + TKM - 1) / TKM : 0;
  return it;
}

template <int TKM>
__device__ __forceinline__ int a_mine(const AItem& it, int warp) {
  return it.ntile > warp ? (it.ntile - warp + MW - 1) / MW : 0;
}

// ---- the per-warp stream of slots (state kept in lane 0) -----------------------------------
// The producer lane walks every phase q = layer * kPhases + j (then the lm_head
// phase) in order; enter() caches where the current phase's copies come from.
template <int D, typename KVT>
struct Stream {
  static constexpr int TKM = tile_keys<D, KVT>();
  static constexpr int ROWB = D * sizeof(KVT);
  static constexpr bool I8 = std::is_same<KVT, int8_t>::value;
  int q = 0, k = 0, n = 0, issued = 0, lastq = 0;
  bool done = false, attn = false;
  const uint8_t* src = nullptr;  // GEMV: next unit to copy
  int left = 0;                  // GEMV: units still to copy
  const uint8_t* kb = nullptr;   // attention: K / V rows and scales of this KV head
  const uint8_t* vb = nullptr;
  const __half* ksb = nullptr;
  const __half* vsb = nullptr;
  int j0 = 0, k1 = 0;

  __device__ void enter(const MegaArgs& a, int cta, int G, int warp, int pos, int qkv_n) {
    k = 0;
    n = 0;
    attn = false;
    if (q > lastq) return;
    const int l = q / kPhases, j = q - (q / kPhases) * kPhases;
    if (l < a.n_layers && j == PH_MERGE) return;
    if (l < a.n_layers && j == PH_ATTN) {
      if (cta >= a.nkv * a.nsplit) return;
      const AItem it = a_item<TKM>(a, cta, pos + 1);
      const LayerPtrs& lp = a.layers[l];
      const size_t head_row = (static_cast<size_t>(a.seq) * a.nkv + it.g) * a.cap;
      attn = true;
      n = a_mine<TKM>(it, warp);
      kb = static_cast<const uint8_t*>(lp.kc) + head_row * ROWB;
      vb = static_cast<const uint8_t*>(lp.vc) + head_row * ROWB;
      if constexpr (I8) {
        ksb = static_cast<const __half*>(lp.ks) + head_row;
        vsb = static_cast<const __half*>(lp.vs) + head_row;
      }
      j0 = it.k0 + warp * TKM;
      k1 = it.k1;
      return;
    }
    const GDesc d = gdesc(a, q, qkv_n, D);
    const GRange r = g_range(d, cta, G, warp);
    n = r.nslots;
    src = d.W + (static_cast<size_t>(r.p0) * d.CT + r.ua) * kUnit;
    left = r.ub - r.ua;
  }

  // advance to the next phase that has slots for this warp
  __device__ void next_phase(const MegaArgs& a, int cta, int G, int warp, int pos, int qkv_n) {
    while (n == 0 && q <= lastq) {
      ++q;
      enter(a, cta, G, warp, pos, qkv_n);
    }
    done = q > lastq;
  }

  __device__ void start(const MegaArgs& a, uint8_t* ring, uint64_t* full, int cta, int G, int warp, int pos,
                        int qkv_n) {
    lastq = a.n_layers * kPhases - 1 + (a.head ? 1 : 0);
    q = 0;
    issued = 0;
    enter(a, cta, G, warp, pos, qkv_n);
    next_phase(a, cta, G, warp, pos, qkv_n);
    for (int i = 0; i < NS; ++i) issue_next(a, ring, full, cta, G, warp, pos, qkv_n);
  }

  __device__ void issue_next(const MegaArgs& a, uint8_t* ring, uint64_t* full, int cta, int G, int warp, int pos,
                             int qkv_n) {
    if (done) return;
    const int s = issued % NS;
    uint8_t* dst = ring + static_cast<size_t>(s) * SB;
    uint64_t* bar = &full[s];
    if (attn) {
      const int rows = min(TKM, k1 - j0);
      const int crow = max(0, min(rows, pos - j0));  // cached rows; row pos is written this step
      const int srow = (crow + 7) & ~7;
      const uint32_t bytes = 2u * crow * ROWB + (I8 && crow > 0 ? 2u * srow * 2u : 0u);
      if (bytes == 0) {
        mbar_arrive(bar);
      } else {
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(dst, kb + static_cast<size_t>(j0) * ROWB, crow * ROWB, bar);
        bulk_g2s(dst + TKM * ROWB, vb + static_cast<size_t>(j0) * ROWB, crow * ROWB, bar);
        if constexpr (I8) {
          bulk_g2s(dst + 2 * TKM * ROWB, ksb + j0, srow * 2u, bar);
          bulk_g2s(dst + 2 * TKM * ROWB + TKM * 2, vsb + j0, srow * 2u, bar);
        }
      }
      j0 += MW * TKM;
    } else {
      const int nu = min(SU, left);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nu) * kUnit);
      bulk_g2s(dst, src, static_cast<uint32_t>(nu) * kUnit, bar);
      src += static_cast<size_t>(nu) * kUnit;
      left -= nu;
    }
    ++issued;
    if (++k >= n) {
      n = 0;
      next_phase(a, cta, G, warp, pos, qkv_n);
    }
  }
};

struct GEpi {
  int epi;  // EPI_QKV, EPI_RESID, EPI_SWIGLU or EPI_ARGMAX
  float* out;
  const float2* rope;
  int pos;
  int head_dim;
  int n_rot;
  float* logits;
  float* resid_init;  // layer 0: CTA 0 stores the raw embedding row here
  unsigned* guard;
};

template <typename WT>
__device__ __forceinline__ float4 load4_weight(const WT* p, int e);
template <>
__device__ __forceinline__ float4 load4_weight<__nv_bfloat16>(const __nv_bfloat16* p, int e) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(p + e));
  return make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
}
template <>
__device__ __forceinline__ float4 load4_weight<float>(const float* p, int e) {
  return __ldg(reinterpret_cast<const float4*>(p + e));
}

// One GEMV phase: rebuild x in shared memory, then consume this warp's slots
// (already in flight) and refill the ring from the stream.  x comes from xg
// (fp32, written by an earlier phase) or from xe (an embedding row).
template <typename WT, int D, typename KVT>
__device__ bool g_phase(const MegaArgs& a, const GDesc& d, const float* xg, const WT* xe, const GEpi& ep,
                        uint8_t* smem, MegaShared& sh, Stream<D, KVT>& st, int& consumed, Best& best, int cta, int G,
                        int pos, int qkv_n) {
  constexpr int EPL = Unpack<WT>::N;
  constexpr int CH = 32 * EPL;
  constexpr int NPL = EPL / 4;
  constexpr int PX = 10;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = d.K, CT = d.CT;
  float* xs = reinterpret_cast<float*>(smem + kMegaRingBytes);
  uint8_t* ring = smem + static_cast<size_t>(warp) * NS * SB;
  const GRange r = g_range(d, cta, G, warp);
  if (lane == 0) sh.rec_n[warp] = 0;

  // ---- x, normalised if the phase has a gain, lane-interleaved per chunk
  {
    const int KP = CT * CH;
    const int gsz = d.gain ? K / a.groups : K;
    auto xidx = [&](int e) {
      const int c = e / CH, rr = e - c * CH, l = rr / EPL, j = rr - l * EPL;
      return ((c * NPL + j / 4) * 32 + l) * 4;
    };
    auto load4 = [&](int e) -> float4 {
      if (e >= K) return make_float4(0.f, 0.f, 0.f, 0.f);
      if (xg) return __ldcg(reinterpret_cast<const float4*>(xg + e));
      return load4_weight<WT>(xe, e);
    };
    float ssq[4] = {0.f, 0.f, 0.f, 0.f};
    auto add_ssq = [&](int e, float4 v) {
      const float t = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      const int grp = e < K ? e / gsz : 4;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q == grp) ssq[q] += t;
    };
    // everything this phase reads from L2 is requested at once: x, the gain,
    // and the epilogue's residual rows or RoPE factors
    constexpr int PG = 4;  // float4s of the gain per thread held in registers (K <= 4096)
    const WT* gw = static_cast<const WT*>(d.gain);
    float side = 0.f;
    float2 side2 = make_float2(1.f, 0.f);
    if (ep.epi == EPI_RESID) {
      if (tid < min(2 * r.p1, d.N) - 2 * r.p0) side = __ldcg(ep.out + 2 * r.p0 + tid);
    } else if (ep.epi == EPI_QKV) {
      const int half = ep.head_dim / 2;
      const int g = r.p0 + tid;
      if (g < r.p1 && g / half < ep.n_rot) side2 = ep.rope[static_cast<size_t>(ep.pos) * half + (g - (g / half) * half)];
    }
    float4 gq[PG];
#pragma unroll
    for (int i = 0; i < PG; ++i) {
      const int e = tid * 4 + i * MT * 4;
      gq[i] = (gw != nullptr && e < K) ? load4_weight<WT>(gw, e) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 xq[PX];
#pragma unroll
    for (int i = 0; i < PX; ++i) xq[i] = load4(tid * 4 + i * MT * 4);
    if (ep.epi == EPI_RESID) {
      if (tid < 2 * kMegaPairsMax) sh.rsd[tid] = side;
    } else if (ep.epi == EPI_QKV) {
      if (tid < kMegaPairsMax) sh.rope[tid] = side2;
    }
#pragma unroll
    for (int i = 0; i < PX; ++i) add_ssq(tid * 4 + i * MT * 4, xq[i]);
    for (int e = tid * 4 + PX * MT * 4; e < KP; e += MT * 4) {
      const float4 v = load4(e);
      *reinterpret_cast<float4*>(xs + xidx(e)) = v;
      add_ssq(e, v);
    }
    if (ep.resid_init && cta == 0) {
#pragma unroll
      for (int i = 0; i < PX; ++i) {
        const int e = tid * 4 + i * MT * 4;
        if (e < K) __stcg(reinterpret_cast<float4*>(ep.resid_init + e), xq[i]);
      }
      for (int e = tid * 4 + PX * MT * 4; e < K; e += MT * 4)
        __stcg(reinterpret_cast<float4*>(ep.resid_init + e), load4(e));
    }
    if (d.gain != nullptr) {
#pragma unroll
      for (int q = 0; q < 4; ++q) ssq[q] = warp_sum(ssq[q]);
      if (lane == 0)
        for (int q = 0; q < 4; ++q) sh.ss[warp][q] = ssq[q];
      __syncthreads();
      if (tid < a.groups) {
        float t = 0.f;
        for (int w = 0; w < MW; ++w) t += sh.ss[w][tid];
        sh.rs[tid] = 1.0f / sqrtf(t / static_cast<float>(gsz) + a.eps);
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < PX; ++i) {
        const int e = tid * 4 + i * MT * 4;
        if (e < KP) {
          float4 v = xq[i];
          if (e < K) {
            const float rs = sh.rs[e / gsz];
            const float4 gn = i < PG ? gq[i < PG ? i : 0] : load4_weight<WT>(gw, e);
            v.x = v.x * rs * gn.x; v.y = v.y * rs * gn.y; v.z = v.z * rs * gn.z; v.w = v.w * rs * gn.w;
          }
          *reinterpret_cast<float4*>(xs + xidx(e)) = v;
        }
      }
      for (int e = tid * 4 + PX * MT * 4; e < K; e += MT * 4) {
        float4* q = reinterpret_cast<float4*>(xs + xidx(e));
        const float rs = sh.rs[e / gsz];
        const float4 gn = load4_weight<WT>(gw, e);
        float4 v = *q;
        v.x = v.x * rs * gn.x; v.y = v.y * rs * gn.y; v.z = v.z * rs * gn.z; v.w = v.w * rs * gn.w;
        *q = v;
      }
    } else {
#pragma unroll
      for (int i = 0; i < PX; ++i) {
        const int e = tid * 4 + i * MT * 4;
        if (e < KP) *reinterpret_cast<float4*>(xs + xidx(e)) = xq[i];
      }
    }
    __syncthreads();
  }

  auto finish = [&](int g, float v0, float v1) {
    const int row = 2 * g;
    if (ep.epi == EPI_SWIGLU) {
      __stcg(ep.out + g, v0 / (1.0f + expf(-v0)) * v1);
    } else if (ep.epi == EPI_QKV) {
      const int half = ep.head_dim / 2;
      const int head = g / half, i = g - head * half;
      float o0 = v0, o1 = v1;
      if (head < ep.n_rot) {
        const float2 cs = sh.rope[g - r.p0];
        o0 = v0 * cs.x - v1 * cs.y;
        o1 = v1 * cs.x + v0 * cs.y;
      }
      __stcg(ep.out + head * ep.head_dim + i, o0);
      __stcg(ep.out + head * ep.head_dim + i + half, o1);
    } else {
      const int rows = min(2, d.N - row);
      const float v[2] = {v0, v1};
      for (int rr = 0; rr < rows; ++rr) {
        if (ep.epi == EPI_RESID) {
          __stcg(ep.out + row + rr, sh.rsd[row + rr - 2 * r.p0] + v[rr]);
        } else {
          if (ep.logits) ep.logits[row + rr] = v[rr];
          if (v[rr] != v[rr]) atomicOr(ep.guard, GUARD_NAN);
          else best = better(best, Best{v[rr], row + rr});
        }
      }
    }
  };

  int pl = r.ua / CT, c = r.ua - (r.ua / CT) * CT;
  bool pair_whole = (c == 0);
  float acc0 = 0.f, acc1 = 0.f;
  bool bad = false;
  for (int k = 0; k < r.nslots; ++k) {
    const int s = consumed % NS;
    const bool ok = mbar_wait(&sh.full[warp][s], static_cast<uint32_t>(consumed / NS) & 1u);
    if (__any_sync(0xffffffffu, !ok)) {
      bad = true;
      break;
    }
    const uint8_t* buf = ring + static_cast<size_t>(s) * SB;
    const int u0 = r.ua + k * SU;
    const int n = min(SU, r.ub - u0);
    int j = 0;
    while (j < n) {
      const int seg = min(n - j, CT - c);
#pragma unroll 2
      for (int q = 0; q < seg; ++q) {
        const int cc = c + q;
        float xv[EPL];
#pragma unroll
        for (int pp = 0; pp < NPL; ++pp) {
          const float4 t = *reinterpret_cast<const float4*>(xs + ((cc * NPL + pp) * 32 + lane) * 4);
          xv[4 * pp] = t.x; xv[4 * pp + 1] = t.y; xv[4 * pp + 2] = t.z; xv[4 * pp + 3] = t.w;
        }
        const uint8_t* u8 = buf + (j + q) * kUnit + lane * 16;
        float w0[EPL], w1[EPL];
        Unpack<WT>::run(*reinterpret_cast<const uint4*>(u8), w0);
        Unpack<WT>::run(*reinterpret_cast<const uint4*>(u8 + 512), w1);
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
      const bool range_end = (u0 + j == r.ub);
      if (pair_end || range_end) {
        const float s0 = warp_sum(acc0), s1 = warp_sum(acc1);
        acc0 = acc1 = 0.f;
        if (lane == 0) {
          if (pair_whole && pair_end) {
            finish(r.p0 + pl, s0, s1);
          } else {
            const int rr = sh.rec_n[warp];
            sh.rec_pair[warp][rr] = pl;
            sh.rec_val[warp][rr][0] = s0;
            sh.rec_val[warp][rr][1] = s1;
            sh.rec_n[warp] = rr + 1;
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
    ++consumed;
    if (lane == 0) {
      fence_proxy_async();
      st.issue_next(a, smem + static_cast<size_t>(warp) * NS * SB, sh.full[warp], cta, G, warp, pos, qkv_n);
    }
  }
  if (bad && lane == 0) atomicOr(a.guard, GUARD_TIMEOUT);
  __syncthreads();
  if (tid == 0) {
    int cur = -1;
    float v0 = 0.f, v1 = 0.f;
    for (int w = 0; w < MW; ++w) {
      for (int rr = 0; rr < sh.rec_n[w]; ++rr) {
        if (sh.rec_pair[w][rr] != cur) {
          if (cur >= 0) finish(r.p0 + cur, v0, v1);
          cur = sh.rec_pair[w][rr];
          v0 = v1 = 0.f;
        }
        v0 += sh.rec_val[w][rr][0];
        v1 += sh.rec_val[w][rr][1];
      }
    }
    if (cur >= 0) finish(r.p0 + cur, v0, v1);
  }
  return __syncthreads_and(!bad) != 0;
}

// ---- attention phase ------------------------------------------------------------------------
template <int DPL>
__device__ __forceinline__ void vload(const float* p, float* f) {
#pragma unroll
  for (int i = 0; i < DPL; ++i) f[i] = p[i];
}
template <int DPL>
__device__ __forceinline__ void vload(const __half* p, float* f) {
  if constexpr (DPL % 2 == 0) {
#pragma unroll
    for (int i = 0; i < DPL; i += 2) {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(p + i));
      f[i] = t.x;
      f[i + 1] = t.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < DPL; ++i) f[i] = __half2float(p[i]);
  }
}
template <int DPL>
__device__ __forceinline__ void vload(const int8_t* p, float* f) {
#pragma unroll
  for (int i = 0; i < DPL; ++i) f[i] = static_cast<float>(p[i]);
}

template <typename WT, int D, int REP, typename KVT>
__device__ bool a_phase(const MegaArgs& a, int l, int pos, uint8_t* smem, MegaShared& sh, Stream<D, KVT>& st,
                        int& consumed, int cta, int G, int qkv_n) {
  constexpr int ELT = sizeof(KVT);
  constexpr int EPL = 16 / ELT;
  constexpr int ROWB = D * ELT;
  constexpr int NV = ROWB / 16;
  constexpr int LPK = NV >= 8 ? 8 : NV;
  constexpr int VPL = NV / LPK;
  constexpr int KPS = 32 / LPK;
  constexpr int QD = VPL * EPL;
  constexpr int DPL = D >= 32 ? D / 32 : 1;
  constexpr int DL = D / DPL;
  constexpr bool I8 = std::is_same<KVT, int8_t>::value;
  constexpr int TKM = tile_keys<D, KVT>();
  constexpr uint32_t KVB = TKM * ROWB;
  constexpr int PSTR = REP * (D + 2);
  static_assert(TKM > 0 && 2 * KVB + 2 * TKM * 2 <= SB, "an attention tile must fit one slot");
  static_assert(D <= 128, "the new K/V rows are staged in a 128-float buffer");
  __shared__ float Sw[MW][REP][TKM];
  __shared__ __align__(16) float Pw[MW][TKM][REP];
  __shared__ float wstate[MW][PSTR];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (cta >= a.nkv * a.nsplit) return true;
  const int L = pos + 1;
  const AItem it = a_item<TKM>(a, cta, L);
  const int nmine = a_mine<TKM>(it, warp);
  const LayerPtrs& lp = a.layers[l];
  const size_t head_row = (static_cast<size_t>(a.seq) * a.nkv + it.g) * a.cap;
  uint8_t* ring = smem + static_cast<size_t>(warp) * NS * SB;
  const float* qkv = a.qkv;
  const int kl = lane % LPK;
  float q[REP][QD];
#pragma unroll
  for (int h = 0; h < REP; ++h)
#pragma unroll
    for (int e = 0; e < QD; ++e) q[h][e] = __ldcg(qkv + (it.g * REP + h) * D + kl * QD + e) * a.scale;
  // the CTA holding the last keys appends the new token: stage its K and V
  // rows now, in the same round trip as q
  if (it.k1 == L) {
    for (int idx = tid; idx < 2 * D; idx += MT) {
      const int kv = idx / D, e = idx - (idx / D) * D;
      sh.newkv[kv][e] = __ldcg(qkv + (kv == 0 ? a.nq * D : (a.nq + a.nkv) * D) + it.g * D + e);
    }
  }
  __syncthreads();

  float m[REP], lsum[REP], acc[REP][DPL];
#pragma unroll
  for (int h = 0; h < REP; ++h) {
    m[h] = -INFINITY;
    lsum[h] = 0.f;
#pragma unroll
    for (int dd = 0; dd < DPL; ++dd) acc[h][dd] = 0.f;
  }
  bool bad = false;
  for (int i = 0; i < nmine; ++i) {
    const int t = warp + i * MW;
    const int j0 = it.k0 + t * TKM;
    const int rows = min(TKM, it.k1 - j0);
    const int s = consumed % NS;
    const bool ok = mbar_wait(&sh.full[warp][s], static_cast<uint32_t>(consumed / NS) & 1u);
    if (__any_sync(0xffffffffu, !ok)) {
      bad = true;
      break;
    }
    uint8_t* slot = ring + static_cast<size_t>(s) * SB;
    const __half* ksc = reinterpret_cast<const __half*>(slot + 2 * KVB);
    const __half* vsc = ksc + TKM;
    const int jr = pos - j0;
    if (it.k1 == L && jr >= 0 && jr < rows) {  // the new token: cache format, to global and into the slot
      for (int kv = 0; kv < 2; ++kv) {
        const float* src = sh.newkv[kv];
        KVT* dst = static_cast<KVT*>(kv == 0 ? lp.kc : lp.vc) + (head_row + pos) * D;
        KVT* row = reinterpret_cast<KVT*>(slot + kv * KVB + jr * ROWB);
        if constexpr (I8) {
          float amax = 0.f;
          for (int e = lane; e < D; e += 32) amax = fmaxf(amax, fabsf(src[e]));
          amax = warp_max(amax);
          const __half sh16 = __float2half_rn(fminf(amax / 127.0f, 65504.0f));
          const float sf = __half2float(sh16);
          for (int e = lane; e < D; e += 32) {
            float cq = sf > 0.f ? rintf(src[e] / sf) : 0.f;
            cq = fminf(fmaxf(cq, -127.f), 127.f);
            const int8_t ci = static_cast<int8_t>(cq);
            dst[e] = ci;
            row[e] = ci;
          }
          if (lane == 0) {
            static_cast<__half*>(kv == 0 ? lp.ks : lp.vs)[head_row + pos] = sh16;
            reinterpret_cast<__half*>(slot + 2 * KVB + kv * TKM * 2)[jr] = sh16;
          }
        } else if constexpr (std::is_same<KVT, __half>::value) {
          for (int e = lane; e < D; e += 32) {
            const __half hv = __float2half_rn(src[e]);
            dst[e] = hv;
            row[e] = hv;
          }
        } else {
          for (int e = lane; e < D; e += 32) {
            const float v = src[e];
            dst[e] = v;
            row[e] = v;
          }
        }
      }
      __syncwarp();
    }
#pragma unroll
    for (int stp = 0; stp < (TKM + KPS - 1) / KPS; ++stp) {
      const int jj = stp * KPS + lane / LPK;
      float dot[REP];
#pragma unroll
      for (int h = 0; h < REP; ++h) dot[h] = 0.f;
      if (jj < rows) {
        const uint8_t* kr = slot + jj * ROWB + kl * VPL * 16;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          float kf[EPL];
          Unpack<KVT>::run(*reinterpret_cast<const uint4*>(kr + v * 16), kf);
#pragma unroll
          for (int h = 0; h < REP; ++h)
#pragma unroll
            for (int e = 0; e < EPL; ++e) dot[h] = fmaf(q[h][v * EPL + e], kf[e], dot[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < REP; ++h)
#pragma unroll
        for (int o = LPK / 2; o > 0; o >>= 1) dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], o);
      if (kl == 0 && jj < rows) {
        const float sc = I8 ? __half2float(ksc[jj]) : 1.f;
#pragma unroll
        for (int h = 0; h < REP; ++h) Sw[warp][h][jj] = dot[h] * sc;
      }
    }
    __syncwarp();
    float al[REP];
#pragma unroll
    for (int h = 0; h < REP; ++h) {
      const float sv = lane < rows ? Sw[warp][h][lane] : -INFINITY;
      const float mn = fmaxf(m[h], warp_max(sv));
      al[h] = expf(m[h] - mn);
      const float pr = lane < rows ? expf(sv - mn) : 0.f;
      lsum[h] = lsum[h] * al[h] + warp_sum(pr);
      m[h] = mn;
      if (lane < rows) Pw[warp][lane][h] = I8 ? pr * __half2float(vsc[lane]) : pr;
    }
    __syncwarp();
    if (lane < DL) {
#pragma unroll
      for (int h = 0; h < REP; ++h)
#pragma unroll
        for (int dd = 0; dd < DPL; ++dd) acc[h][dd] *= al[h];
      const KVT* vt = reinterpret_cast<const KVT*>(slot + KVB) + lane * DPL;
      for (int jj = 0; jj < rows; ++jj) {
        float vf[DPL];
        vload<DPL>(vt + jj * D, vf);
        float pr[REP];
        if constexpr (REP == 4) {
          const float4 p4 = *reinterpret_cast<const float4*>(&Pw[warp][jj][0]);
          pr[0] = p4.x; pr[1] = p4.y; pr[2] = p4.z; pr[3] = p4.w;
        } else {
#pragma unroll
          for (int h = 0; h < REP; ++h) pr[h] = Pw[warp][jj][h];
        }
#pragma unroll
        for (int h = 0; h < REP; ++h)
#pragma unroll
          for (int dd = 0; dd < DPL; ++dd) acc[h][dd] = fmaf(pr[h], vf[dd], acc[h][dd]);
      }
    }
    // the slot may have been written here (the new row): order those generic
    // writes, and every lane's reads, before the next bulk copy into it
    fence_proxy_async();
    __syncwarp();
    ++consumed;
    if (lane == 0) st.issue_next(a, ring, sh.full[warp], cta, G, warp, pos, qkv_n);
  }
  if (bad && lane == 0) atomicOr(a.guard, GUARD_TIMEOUT);
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < REP; ++h) {
      wstate[warp][h] = m[h];
      wstate[warp][REP + h] = lsum[h];
    }
  }
  if (lane < DL) {
#pragma unroll
    for (int h = 0; h < REP; ++h)
#pragma unroll
      for (int dd = 0; dd < DPL; ++dd) wstate[warp][2 * REP + h * D + lane * DPL + dd] = acc[h][dd];
  }
  __syncthreads();
  float* pp = a.part + static_cast<size_t>(cta) * PSTR;
  for (int idx = tid; idx < REP * D; idx += MT) {
    const int h = idx / D;
    float M = -INFINITY;
    for (int w = 0; w < MW; ++w) M = fmaxf(M, wstate[w][h]);
    float O = 0.f;
    for (int w = 0; w < MW; ++w)
      if (wstate[w][h] != -INFINITY) O = fmaf(wstate[w][2 * REP + idx], expf(wstate[w][h] - M), O);
    __stcg(pp + 2 * REP + idx, O);
  }
  if (tid < REP) {
    float M = -INFINITY;
    for (int w = 0; w < MW; ++w) M = fmaxf(M, wstate[w][tid]);
    float Ls = 0.f;
    for (int w = 0; w < MW; ++w)
      if (wstate[w][tid] != -INFINITY) Ls = fmaf(wstate[w][REP + tid], expf(wstate[w][tid] - M), Ls);
    __stcg(pp + tid, M);
    __stcg(pp + REP + tid, Ls);
  }
  return __syncthreads_and(!bad) != 0;
}

// outputs [cta * chunk, ...) of all query heads: log-sum-exp merge of the splits
template <int D, int REP>
__device__ void merge_phase(const MegaArgs& a, int cta, int G) {
  constexpr int PSTR = REP * (D + 2);
  const int total = a.nq * D;
  const int chunk = (total + G - 1) / G;
  const int lo = cta * chunk, hi = min(total, lo + chunk);
  const int ns = a.nsplit;
  for (int idx = lo + static_cast<int>(threadIdx.x); idx < hi; idx += MT) {
    const int qh = idx / D, dd = idx - qh * D;
    const int g = qh / REP, h = qh - g * REP;
    const float* base = a.part + static_cast<size_t>(g) * ns * PSTR;
    // one pass over the splits, rescaling as the running maximum grows
    float M = -INFINITY, Ls = 0.f, O = 0.f;
#pragma unroll 4
    for (int s = 0; s < ns; ++s) {
      const float ms = __ldcg(base + s * PSTR + h);
      const float ls = __ldcg(base + s * PSTR + REP + h);
      const float os = __ldcg(base + s * PSTR + 2 * REP + h * D + dd);
      if (ms == -INFINITY) continue;
      const float mn = fmaxf(M, ms);
      const float wo = expf(M - mn), ws = expf(ms - mn);
      Ls = Ls * wo + ls * ws;
      O = O * wo + os * ws;
      M = mn;
    }
    __stcg(a.attn_out + idx, O / Ls);
  }
}

// ---- the step -------------------------------------------------------------------------------
template <typename WT, int D, int REP, typename KVT>
__global__ void __launch_bounds__(MT, 1) mega_decode_kernel(const MegaArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ MegaShared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  const int pos = a.seq_len[a.seq];
  if (pos < 0 || pos >= a.cap) {
    if (tid == 0) atomicOr(a.guard, GUARD_POS);
    return;  // every CTA sees the same pos and leaves before any grid barrier
  }
  const int qkv_n = (a.nq + 2 * a.nkv) * D;
  Stream<D, KVT> st;
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&sh.full[warp][s], 1);
    fence_mbar_init();
    st.start(a, smem + static_cast<size_t>(warp) * NS * SB, sh.full[warp], cta, G, warp, pos, qkv_n);
  }
  __syncwarp();
  int consumed = 0;
  Best best{-INFINITY, 0x7fffffff};

  const WT* xe = nullptr;
  if (!a.x_ext) {
    const int tok = *a.token_in;
    if (tok < 0 || tok >= a.vocab) {
      if (tid == 0) atomicOr(a.guard, GUARD_TOKEN);
      xe = static_cast<const WT*>(a.embed);  // row 0 stands in; the guard reports the fault
    } else {
      xe = static_cast<const WT*>(a.embed) + static_cast<size_t>(tok) * a.hidden;
    }
  }
  float* resid = a.x_ext ? a.x_ext : a.resid;

  // One loop over the phases, so that each phase body exists once in the
  // code: the instruction cache stays warm from one phase to the next.
  const int lastq = a.n_layers * kPhases - 1 + (a.head ? 1 : 0);
  bool ok = true;
  for (int q = 0; q <= lastq; ++q) {
    const int l = q / kPhases, j = q - (q / kPhases) * kPhases;
    if (l < a.n_layers && j == PH_ATTN) {
      ok = a_phase<WT, D, REP>(a, l, pos, smem, sh, st, consumed, cta, G, qkv_n);
    } else if (l < a.n_layers && j == PH_MERGE) {
      merge_phase<D, REP>(a, cta, G);
    } else {
      GEpi ep{EPI_RESID, resid, a.rope, pos, D, a.nq + a.nkv, nullptr, nullptr, a.guard};
      const float* xg = resid;
      const WT* xr = nullptr;
      if (l >= a.n_layers) {
        ep.epi = EPI_ARGMAX;
        ep.out = nullptr;
        ep.logits = a.logits;
      } else if (j == PH_QKV) {
        ep.epi = EPI_QKV;
        ep.out = a.qkv;
        if (l == 0) {
          xg = a.x_ext;
          xr = xe;
          if (!a.x_ext) ep.resid_init = resid;
        }
      } else if (j == PH_O) {
        xg = a.attn_out;
      } else if (j == PH_GU) {
        ep.epi = EPI_SWIGLU;
        ep.out = a.act;
      } else {
        xg = a.act;
      }
      ok = g_phase<WT, D, KVT>(a, gdesc(a, q, qkv_n, D), xg, xr, ep, smem, sh, st, consumed, best, cta, G, pos,
                               qkv_n);
    }
    if (!ok) break;
    if (q < lastq && !grid_sync(a, sh, q)) {
      ok = false;
      break;
    }
  }
  if (ok && a.head) {
    best = warp_best(best);
    if (lane == 0) sh.best[warp] = best;
    __syncthreads();
    if (tid == 0) {
      Best b = sh.best[0];
      for (int w = 1; w < MW; ++w) b = better(b, sh.best[w]);
      __stcg(a.am_val + cta, b.v);
      __stcg(a.am_idx + cta, b.i);
    }
  }
  // On a failed wait some copies of this warp may still be in flight: wait
  // (bounded) for them before the CTA's shared memory goes away.
  if (lane == 0) {
    for (; consumed < st.issued; ++consumed)
      if (!mbar_wait(&sh.full[warp][consumed % NS], static_cast<uint32_t>(consumed / NS) & 1u)) break;
  }
  // the last CTA to get here finishes the step and re-arms the barrier
  // counters (every CTA is past its last grid barrier by then)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned t = atomicAdd(a.end_count, 1u);
    sh.flag = (t == static_cast<unsigned>(G - 1));
  }
  __syncthreads();
  if (!sh.flag) return;
  __threadfence();
  const bool failed = (__ldcg(a.guard) & GUARD_TIMEOUT) != 0u;
  if (a.head && !failed) {
    Best b{-INFINITY, 0x7fffffff};
    for (int i = tid; i < G; i += MT) b = better(b, Best{__ldcg(a.am_val + i), __ldcg(a.am_idx + i)});
    b = warp_best(b);
    if (lane == 0) sh.best[warp] = b;
    __syncthreads();
    if (tid == 0) {
      Best f = sh.best[0];
      for (int w = 1; w < MW; ++w) f = better(f, sh.best[w]);
      if (f.i == 0x7fffffff) {
        atomicOr(a.guard, GUARD_NAN);
        f.i = 0;
      }
      *a.token_out = f.i;
    }
  }
  if (tid == 0) {
    if (!failed) a.seq_len[a.seq] = pos + 1;
    *a.bar_count = 0u;
    *a.end_count = 0u;
  }
}

template <int D, typename KVT>
constexpr bool tile_fits() {
  return tile_keys<D, KVT>() > 0;
}

template <typename WT, int D, int REP, typename KVT>
const void* mega_fn() {
  if constexpr (tile_fits<D, KVT>())
    return reinterpret_cast<const void*>(mega_decode_kernel<WT, D, REP, KVT>);
  else
    return nullptr;
}

// (weight type, head_dim, GQA ratio) combinations with a persistent kernel:
// the 3.7B shape, the medium and the tiny test models
#define K2_MEGA_SHAPES(X) X(__nv_bfloat16, 2, 128, 4) X(__nv_bfloat16, 2, 64, 4) X(float, 4, 16, 2)

const void* mega_lookup(int wbytes, int head_dim, int rep, int kv_dtype) {
#define K2_MEGA_LOOK(WT, WB, D, R)                                  \
  if (wbytes == WB && head_dim == D && rep == R) {                  \
    if (kv_dtype == 0) return mega_fn<WT, D, R, float>();           \
    if (kv_dtype == 2) return mega_fn<WT, D, R, __half>();          \
    if (kv_dtype == 3) return mega_fn<WT, D, R, int8_t>();          \
  }
  K2_MEGA_SHAPES(K2_MEGA_LOOK)
#undef K2_MEGA_LOOK
  return nullptr;
}

}  // namespace

bool mega_supported(int wbytes, int head_dim, int rep, int kv_dtype) {
  return mega_lookup(wbytes, head_dim, rep, kv_dtype) != nullptr;
}

cudaError_t mega_init_attrs(int wbytes, int head_dim, int rep, int kv_dtype) {
  const void* fn = mega_lookup(wbytes, head_dim, rep, kv_dtype);
  if (!fn) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMegaSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                              static_cast<int>(cudaSharedmemCarveoutMaxShared));
}

int mega_max_grid(int wbytes, int head_dim, int rep, int kv_dtype) {
  const void* fn = mega_lookup(wbytes, head_dim, rep, kv_dtype);
  if (!fn) return 0;
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, MT, kMegaSmemBytes) != cudaSuccess) return 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return per_sm >= 1 ? sms : 0;  // one CTA per SM
}

cudaError_t launch_mega(const MegaArgs& a, int wbytes, int head_dim, int rep, int kv_dtype, int grid, cudaStream_t s) {
  const void* fn = mega_lookup(wbytes, head_dim, rep, kv_dtype);
  if (!fn) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MT);
  cfg.dynamicSmemBytes = kMegaSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<MegaArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace k2
