// Split-K flash-decode GQA attention for one new token per sequence, with the
// KV-cache append of that token fused in.
//
// What it computes (k2-burn README, "Status: v0" GQA attention, "Limitations"
// plain SDPA with an fp32 softmax, "Model shape" 32 q heads over 8 KV heads):
// for query head h of the new token at position pos, with KV head
// g = h / REP, o_h = softmax_j(q_h . k_j / sqrt(D)) . v_j over j = 0..pos.
//
// Layout and schedule:
//   * grid = (splits, KV heads, sequences), and the splits of one (sequence,
//     KV head) form one thread-block cluster; a CTA owns a contiguous key
//     range, so every K/V byte is read from HBM once per step and shared by
//     the REP query heads of the group;
//   * the range is cut into 32-key tiles dealt round-robin to the 4 warps;
//     each warp streams its tiles through its own shared-memory slot with
//     bulk TMA copies (K rows, V rows), the first one requested before
//     griddepcontrol.wait (cached rows never depend on the previous kernel);
//     three CTAs (12 warps) share an SM, so one warp's copy and its
//     latency-bound tile steps overlap the others'; the K and V halves of a
//     slot have their own barriers, so the next tile's K rows are copied
//     while the warp still works on the current tile's softmax and P.V;
//   * per tile a warp computes the 32 scores (8 lanes per key), one fp32
//     online-softmax update (one lane per key) and the P.V product (lanes own
//     output dims), keeping its own (m, l, o) per head: no CTA barrier inside
//     the loop;
//   * the new token's K/V (already rotated by the QKV kernel) are stored in the
//     cache format (fp32, fp16 round-to-nearest, or int8 with one fp16 scale
//     per row, k2-burn README "KV cache storage") by the warp whose tile holds
//     position pos, which also uses the stored values itself;
//   * int8 rows are dequantised inside the kernel (code * row scale);
//   * the warp states are merged in shared memory, then the splits of the
//     cluster merge through distributed shared memory: after a cluster
//     barrier each CTA finalises a slice of the head outputs from its peers'
//     (m, l, o) with log-sum-exp weights -- no partials in global memory, no
//     atomics, no fences.
#include <cuda.h>
#include <math.h>

#include <type_traits>

#include "k2_kernels.h"
#include "k2_common.cuh"

namespace k2 {

namespace {

// element d of head h (q heads, then k, then v) of a token's projections in
// natural order: read as is, or from the QKV GEMM's packed rows (dims i and
// i + D/2 side by side) with q and k rotated by split-half RoPE at position pos
__device__ __forceinline__ float qkv_at(const AttnArgs& a, const float* qkv, int h, int d, int D, int pos) {
  if (a.rope == nullptr) return qkv[h * D + d];
  const int half = D / 2, i = d < half ? d : d - half;
  const float x = qkv[h * D + 2 * i], y = qkv[h * D + 2 * i + 1];
  if (h >= a.nq + a.nkv) return d < half ? x : y;  // v: not rotated
  const float2 cs = a.rope[static_cast<size_t>(pos) * half + i];
  return d < half ? x * cs.x - y * cs.y : y * cs.x + x * cs.y;
}

// the merged output element: fp32 and / or the bf16 hi / lo pair a GEMM takes
__device__ __forceinline__ void store_out(const AttnArgs& a, size_t i, float v) {
  if (a.out != nullptr) a.out[i] = v;
  if (a.out_hi != nullptr) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    a.out_hi[i] = h;
    a.out_lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

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

template <int DPL>
__device__ __forceinline__ void load_dims(const float* p, float* f) {
#pragma unroll
  for (int i = 0; i < DPL; ++i) f[i] = p[i];
}
template <int DPL>
__device__ __forceinline__ void load_dims(const __half* p, float* f) {
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
__device__ __forceinline__ void load_dims(const int8_t* p, float* f) {
#pragma unroll
  for (int i = 0; i < DPL; ++i) f[i] = static_cast<float>(p[i]);
}

// ---- thread-block cluster helpers (distributed shared memory) -----------------
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_peer(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

constexpr int kWarps = kAttnThreads / 32;

template <int D, int REP, typename KVT>
__global__ void __launch_bounds__(kAttnThreads, 3) attn_decode_kernel(const AttnArgs a) {
  constexpr int TK = kAttnTK;
  constexpr int ELT = sizeof(KVT);
  constexpr int EPL = 16 / ELT;              // elements per 16-byte load
  constexpr int ROWB = D * ELT;              // bytes of one K or V row
  constexpr int NV = ROWB / 16;              // 16-byte vectors per row
  constexpr int LPK = NV >= 8 ? 8 : NV;      // lanes sharing one key in the score step
  constexpr int VPL = NV / LPK;              // 16-byte vectors per lane per key
  constexpr int KPS = 32 / LPK;              // keys per score step
  constexpr int QD = VPL * EPL;              // q dims per lane
  constexpr int DPL = D >= 32 ? D / 32 : 1;  // output dims per lane
  constexpr int DL = D / DPL;                // lanes holding output dims
  constexpr bool I8 = KVTraits<KVT>::kI8;
  constexpr uint32_t KVB = TK * ROWB;        // bytes of the K (or V) rows of a tile
  constexpr int PSTR = REP * (D + 2);        // a partial state: m[REP], l[REP], o[REP][D]
  static_assert(NV % LPK == 0 && 32 % LPK == 0 && TK <= 32, "head_dim / dtype");

  extern __shared__ __align__(128) uint8_t smem[];  // kWarps slots of a.slot_bytes
  __shared__ uint64_t fullk[kWarps], fullv[kWarps];  // the K half (+ K scales), the V half (+ V scales)
  __shared__ float Sw[kWarps][REP][TK];
  __shared__ __align__(16) float Pw[kWarps][TK][REP];
  __shared__ float cpart[PSTR];  // this CTA's (m, l, o), read by the cluster peers

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z, g = blockIdx.y, sp = blockIdx.x, ns = gridDim.x;
  const int seq = a.block_mode ? a.block_seq : a.seq0 + b;
  // seq_len was written two or more launches back (see pdl_trigger placement)
  const int pos = a.block_mode ? (a.pos_base_dev ? *a.pos_base_dev : a.pos_base) + b : a.seq_len[seq];
  if (pos < 0 || pos >= a.cap) {
    if (tid == 0) atomicOr(a.guard, GUARD_POS);
    return;  // every CTA of the launch sees the same pos and leaves before any cluster barrier
  }
  const int L = pos + 1;
  const int k0 = min(L, static_cast<int>((static_cast<long long>(L) * sp) / ns) & ~7);
  const int k1 = (sp == ns - 1) ? L : min(L, static_cast<int>((static_cast<long long>(L) * (sp + 1)) / ns) & ~7);
  const int ntile = k1 > k0 ? (k1 - k0 + TK - 1) / TK : 0;
  const int nmine = ntile > warp ? (ntile - warp + kWarps - 1) / kWarps : 0;
  const size_t head_row = (static_cast<size_t>(seq) * a.nkv + g) * a.cap;
  const uint8_t* Kg = reinterpret_cast<const uint8_t*>(a.kc) + head_row * ROWB;
  const uint8_t* Vg = reinterpret_cast<const uint8_t*>(a.vc) + head_row * ROWB;
  const __half* KSg = I8 ? reinterpret_cast<const __half*>(a.ks) + head_row : nullptr;
  const __half* VSg = I8 ? reinterpret_cast<const __half*>(a.vs) + head_row : nullptr;
  uint8_t* slot = smem + static_cast<size_t>(warp) * a.slot_bytes;

  // lane 0: one half (kv = 0: K, 1: V) of tile t of this CTA into this warp's slot
  auto issue = [&](int t, int kv) {
    const int j0 = k0 + t * TK;
    const int rows = min(TK, k1 - j0);
    // cached rows; row pos is the new one (in block mode it is cached too)
    const int crow = max(0, min(rows, (a.block_mode ? pos + 1 : pos) - j0));
    const int srow = (crow + 7) & ~7;             // scale copies in 16-byte units
    uint64_t* bar = kv == 0 ? &fullk[warp] : &fullv[warp];
    const uint32_t bytes = crow * ROWB + (I8 && crow > 0 ? srow * 2u : 0u);
    if (bytes == 0) {
      mbar_arrive(bar);
      return;
    }
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(slot + kv * KVB, (kv == 0 ? Kg : Vg) + static_cast<size_t>(j0) * ROWB, crow * ROWB, bar);
    if constexpr (I8) bulk_g2s(slot + 2 * KVB + kv * TK * 2, (kv == 0 ? KSg : VSg) + j0, srow * 2u, bar);
  };

  if (lane == 0) {
    mbar_init(&fullk[warp], 1);
    mbar_init(&fullv[warp], 1);
    fence_mbar_init();
    if (nmine > 0) {
      issue(warp, 0);
      issue(warp, 1);
    }
  }
  __syncwarp();
  pdl_wait();

  // query slice (pre-scaled by 1/sqrt(D)): dims [kl*QD, kl*QD + QD) of every head
  const float* qkv = a.qkv + static_cast<size_t>(b) * a.qkv_stride;
  const int kl = lane % LPK;
  float q[REP][QD];
#pragma unroll
  for (int h = 0; h < REP; ++h)
#pragma unroll
    for (int e = 0; e < QD; ++e) q[h][e] = qkv_at(a, qkv, g * REP + h, kl * QD + e, D, pos) * a.scale;
  pdl_trigger();

  float m[REP], l[REP], acc[REP][DPL];
#pragma unroll
  for (int h = 0; h < REP; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[h][d] = 0.f;
  }

  bool bad = false;
  int it = 0;
  bool kdone = false, knext = false;  // lane 0: this tile's K half landed; the next tile's K copy issued
  for (; it < nmine; ++it) {
    kdone = knext = false;
    const int t = warp + it * kWarps;
    const int j0 = k0 + t * TK;
    const int rows = min(TK, k1 - j0);
    const uint32_t par = static_cast<uint32_t>(it) & 1u;
    if (__any_sync(0xffffffffu, !mbar_wait(&fullk[warp], par))) {
      bad = true;
      break;
    }
    kdone = true;
    const __half* ksc = reinterpret_cast<const __half*>(slot + 2 * KVB);
    const __half* vsc = ksc + TK;
    // ---- the new token's K/V: stored format to the cache and into the slot
    // (the V half only once its copy has landed)
    const int jr = pos - j0;
    const bool newrow = !a.block_mode && k1 == L && jr >= 0 && jr < rows;
    if (newrow) {
      if (__any_sync(0xffffffffu, !mbar_wait(&fullv[warp], par))) {
        bad = true;
        break;
      }
      for (int kv = 0; kv < 2; ++kv) {
        const int hs = (kv == 0 ? a.nq : a.nq + a.nkv) + g;  // this KV head's k (or v) among the heads
        auto src = [&](int i) { return qkv_at(a, qkv, hs, i, D, pos); };
        KVT* dst = reinterpret_cast<KVT*>(kv == 0 ? a.kc_w : a.vc_w) + (head_row + pos) * D;
        KVT* row = reinterpret_cast<KVT*>(slot + kv * KVB + jr * ROWB);
        if constexpr (I8) {
          float amax = 0.f;
          for (int i = lane; i < D; i += 32) amax = fmaxf(amax, fabsf(src(i)));
          amax = warp_max(amax);
          const __half sh = __float2half_rn(fminf(amax / 127.0f, 65504.0f));
          const float sf = __half2float(sh);
          for (int i = lane; i < D; i += 32) {
            float cq = sf > 0.f ? rintf(src(i) / sf) : 0.f;
            cq = fminf(fmaxf(cq, -127.f), 127.f);
            const int8_t ci = static_cast<int8_t>(cq);
            dst[i] = ci;
            row[i] = ci;
          }
          if (lane == 0) {
            (kv == 0 ? reinterpret_cast<__half*>(a.ks) : reinterpret_cast<__half*>(a.vs))[head_row + pos] = sh;
            reinterpret_cast<__half*>(slot + 2 * KVB + kv * TK * 2)[jr] = sh;
          }
        } else if constexpr (std::is_same<KVT, __half>::value) {
          for (int i = lane; i < D; i += 32) {
            const __half hv = __float2half_rn(src(i));
            dst[i] = hv;
            row[i] = hv;
          }
        } else {
          for (int i = lane; i < D; i += 32) {
            dst[i] = src(i);
            row[i] = src(i);
          }
        }
      }
      __syncwarp();
    }
    // ---- scores: LPK lanes per key, KPS keys per step (keys past the tile: no load, no store)
#pragma unroll
    for (int st = 0; st < (TK + KPS - 1) / KPS; ++st) {
      const int jj = st * KPS + lane / LPK;
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
    // the K half (and K scales) is read: copy the next tile's K rows now
    if (lane == 0 && it + 1 < nmine) {
      if (newrow) fence_proxy_async();  // generic stores into the slot before the bulk copy over them
      issue(t + kWarps, 0);
      knext = true;
    }
    // ---- online softmax: lane j holds key j; every lane keeps the running (m, l)
    float al[REP];
#pragma unroll
    for (int h = 0; h < REP; ++h) {
      const float sv = lane < rows ? Sw[warp][h][lane] : -INFINITY;
      const float mn = fmaxf(m[h], warp_max(sv));
      al[h] = expf(m[h] - mn);  // m = -inf on the first tile: 0, and acc is 0 anyway
      const float p = lane < rows ? expf(sv - mn) : 0.f;
      l[h] = l[h] * al[h] + warp_sum(p);
      m[h] = mn;
      if (lane < rows) Pw[warp][lane][h] = I8 ? p * __half2float(vsc[lane]) : p;
    }
    __syncwarp();
    if (!newrow && __any_sync(0xffffffffu, !mbar_wait(&fullv[warp], par))) {
      bad = true;
      break;
    }
    // ---- o = alpha * o + P . V
    if (lane < DL) {
#pragma unroll
      for (int h = 0; h < REP; ++h)
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[h][d] *= al[h];
      const KVT* vt = reinterpret_cast<const KVT*>(slot + KVB) + lane * DPL;
      for (int j = 0; j < rows; ++j) {
        float vf[DPL];
        load_dims<DPL>(vt + j * D, vf);
        float p[REP];
        if constexpr (REP == 4) {
          const float4 p4 = *reinterpret_cast<const float4*>(&Pw[warp][j][0]);
          p[0] = p4.x; p[1] = p4.y; p[2] = p4.z; p[3] = p4.w;
        } else {
#pragma unroll
          for (int h = 0; h < REP; ++h) p[h] = Pw[warp][j][h];
        }
#pragma unroll
        for (int h = 0; h < REP; ++h)
#pragma unroll
          for (int d = 0; d < DPL; ++d) acc[h][d] = fmaf(p[h], vf[d], acc[h][d]);
      }
    }
    __syncwarp();
    if (lane == 0 && it + 1 < nmine) {
      if (newrow) fence_proxy_async();
      issue(t + kWarps, 1);
    }
  }
  if (bad && lane == 0) {
    atomicOr(a.guard, GUARD_TIMEOUT);
    // the copies that may still be in flight into this slot, bounded: this
    // tile's K half (unless it landed), the next tile's K half (if issued),
    // this tile's V half (a wait that returns at once if it landed)
    const uint32_t par = static_cast<uint32_t>(it) & 1u;
    if (it < nmine) {
      if (!kdone) (void)mbar_wait(&fullk[warp], par);
      if (knext) (void)mbar_wait(&fullk[warp], par ^ 1u);
      (void)mbar_wait(&fullv[warp], par);
    }
  }

  // ---- this warp's state into its (now idle) slot; then the CTA's state -------------
  float* wst = reinterpret_cast<float*>(slot);
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < REP; ++h) {
      wst[h] = m[h];
      wst[REP + h] = l[h];
    }
  }
  if (lane < DL) {
#pragma unroll
    for (int h = 0; h < REP; ++h)
#pragma unroll
      for (int d = 0; d < DPL; ++d) wst[2 * REP + h * D + lane * DPL + d] = acc[h][d];
  }
  __syncthreads();
  for (int idx = tid; idx < REP * D; idx += kAttnThreads) {
    const int h = idx / D;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, reinterpret_cast<const float*>(smem + w * a.slot_bytes)[h]);
    float O = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float* ws = reinterpret_cast<const float*>(smem + w * a.slot_bytes);
      if (ws[h] != -INFINITY) O = fmaf(ws[2 * REP + idx], expf(ws[h] - M), O);
    }
    cpart[2 * REP + idx] = O;
  }
  if (tid < REP) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, reinterpret_cast<const float*>(smem + w * a.slot_bytes)[tid]);
    float Ls = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float* ws = reinterpret_cast<const float*>(smem + w * a.slot_bytes);
      if (ws[tid] != -INFINITY) Ls = fmaf(ws[REP + tid], expf(ws[tid] - M), Ls);
    }
    cpart[tid] = M;
    cpart[REP + tid] = Ls;
  }

  // ---- merge of the cluster's splits through distributed shared memory -------------
  cluster_sync_all();
  const int rank = static_cast<int>(cluster_rank());
  const int chunk = (REP * D + ns - 1) / ns;
  const int lo = rank * chunk, hi = min(REP * D, lo + chunk);
  for (int idx = lo + tid; idx < hi; idx += kAttnThreads) {
    const int h = idx / D;
    float M = -INFINITY;
    for (int s2 = 0; s2 < ns; ++s2) M = fmaxf(M, ld_peer(peer_addr(&cpart[h], s2)));
    float Ls = 0.f, O = 0.f;
    for (int s2 = 0; s2 < ns; ++s2) {
      const float ms = ld_peer(peer_addr(&cpart[h], s2));
      const float w = ms == -INFINITY ? 0.f : expf(ms - M);
      Ls = fmaf(ld_peer(peer_addr(&cpart[REP + h], s2)), w, Ls);
      O = fmaf(ld_peer(peer_addr(&cpart[2 * REP + idx], s2)), w, O);
    }
    store_out(a, static_cast<size_t>(b) * a.nq * D + (g * REP + h) * D + (idx - h * D), O / Ls);
  }
  cluster_sync_all();  // peers read this CTA's cpart until here
}

// ---- tensor-core variant for fp16 caches ------------------------------------------------------
// The same split-K decode attention, with Q.K^T and P.V on the tensor cores:
// mma.sync m16n8k16 (fp16 operands, fp32 accumulation) with the REP query heads
// of the KV head as M rows.  Row h < REP holds fp16(q_h) (or fp16(p_h)), row
// REP + h the remainder q_h - fp16(q_h), so one MMA carries both halves and the
// sum of the two rows keeps about 22 bits of every q and p; the fp16 K/V values
// themselves are exact.  K/V tiles of 32 keys arrive by TMA tensor copies in
// boxes of 64 dims x 32 rows with the 128-byte swizzle (16-byte chunk c of row
// r stored at chunk c ^ (r & 7)), so the ldmatrix fragment loads hit distinct
// banks.  A box always holds 32 rows: rows past the tile's end are masked out of
// the scores and zeroed in V before P.V (stale rows may hold any bit pattern).
template <int D>
struct TcTile {
  static constexpr int NB = D / 64;          // 64-dim boxes per K (or V) tile
  static constexpr int BOX = kAttnTK * 128;  // bytes of one box: 32 rows of 128 B
  static constexpr int KV = NB * BOX;        // bytes of the K (or V) half of a slot
  static constexpr int SLOT = 2 * KV;
};
// byte offset of 16-byte chunk c (0..7) of row r inside a swizzled box
__device__ __forceinline__ uint32_t swz(int r, int c) { return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4)); }
__device__ __forceinline__ void tma_2d_kv(void* dst, const CUtensorMap* m, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(m), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

template <int D, int REP>
__global__ void __launch_bounds__(kAttnThreads, 3) attn_decode_tc_kernel(const __grid_constant__ CUtensorMap mk,
                                                                        const __grid_constant__ CUtensorMap mv,
                                                                        const AttnArgs a) {
  using T = TcTile<D>;
  constexpr int TK = kAttnTK;
  constexpr int KS = D / 16;  // k-steps of Q.K^T
  constexpr int NT = D / 8;   // n-tiles (8 dims) of P.V
  constexpr int PSTR = REP * (D + 2);
  constexpr int XR = 4 * REP;  // lane distance between a head's fp16 row and its remainder row
  static_assert(TK == 32 && D % 64 == 0 && (REP == 1 || REP == 2 || REP == 4), "tile shape");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t fullk[kWarps], fullv[kWarps];
  __shared__ float cpart[PSTR];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;  // fragment row (0..7) and column pair of this lane
  const int hq = gq % REP;                  // the head of this lane's row
  const bool live = gq < 2 * REP, rem = gq >= REP;
  const int b = blockIdx.z, g = blockIdx.y, sp = blockIdx.x, ns = gridDim.x;
  const int seq = a.block_mode ? a.block_seq : a.seq0 + b;
  const int pos = a.block_mode ? (a.pos_base_dev ? *a.pos_base_dev : a.pos_base) + b : a.seq_len[seq];
  if (pos < 0 || pos >= a.cap) {
    if (tid == 0) atomicOr(a.guard, GUARD_POS);
    return;  // every CTA of the launch sees the same pos and leaves before any cluster barrier
  }
  const int L = pos + 1;
  const int k0 = min(L, static_cast<int>((static_cast<long long>(L) * sp) / ns) & ~7);
  const int k1 = (sp == ns - 1) ? L : min(L, static_cast<int>((static_cast<long long>(L) * (sp + 1)) / ns) & ~7);
  const int ntile = k1 > k0 ? (k1 - k0 + TK - 1) / TK : 0;
  const int nmine = ntile > warp ? (ntile - warp + kWarps - 1) / kWarps : 0;
  const size_t head_row = (static_cast<size_t>(seq) * a.nkv + g) * a.cap;
  uint8_t* ksl = smem + static_cast<size_t>(warp) * T::SLOT;
  uint8_t* vsl = ksl + T::KV;

  // lane 0: the K (kv = 0) or V half of tile t, all of its boxes
  auto issue = [&](int t, int kv) {
    const int y = static_cast<int>(head_row) + k0 + t * TK;
    uint64_t* bar = kv == 0 ? &fullk[warp] : &fullv[warp];
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(T::KV));
#pragma unroll
    for (int bx = 0; bx < T::NB; ++bx) tma_2d_kv((kv == 0 ? ksl : vsl) + bx * T::BOX, kv == 0 ? &mk : &mv, 64 * bx, y, bar);
  };

  if (lane == 0) {
    mbar_init(&fullk[warp], 1);
    mbar_init(&fullv[warp], 1);
    fence_mbar_init();
    if (nmine > 0) {
      issue(warp, 0);
      issue(warp, 1);
    }
  }
  __syncwarp();
  pdl_wait();

  // A fragments of the query rows (pre-scaled by 1/sqrt(D)): (a0, a2) per
  // k-step; rows 8..15 (a1, a3) are zero
  const float* qkv = a.qkv + static_cast<size_t>(b) * a.qkv_stride;
  uint32_t qa[KS][2];
  {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int d = 16 * ks + 8 * hf + 2 * tq;
        uint32_t hi = 0u, lo = 0u;
        if (live)
          split_half2(qkv_at(a, qkv, g * REP + hq, d, D, pos) * a.scale,
                      qkv_at(a, qkv, g * REP + hq, d + 1, D, pos) * a.scale, hi, lo);
        qa[ks][hf] = rem ? lo : hi;
      }
  }
  pdl_trigger();

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;

  bool bad = false;
  int it = 0;
  bool kdone = false, knext = false;
  for (; it < nmine; ++it) {
    kdone = knext = false;
    const int t = warp + it * kWarps;
    const int j0 = k0 + t * TK;
    const int rows = min(TK, k1 - j0);
    const uint32_t par = static_cast<uint32_t>(it) & 1u;
    if (__any_sync(0xffffffffu, !mbar_wait(&fullk[warp], par))) {
      bad = true;
      break;
    }
    kdone = true;
    // ---- the new token's K/V: fp16 to the cache and into the (swizzled) slot
    const int jr = pos - j0;
    const bool newrow = !a.block_mode && k1 == L && jr >= 0 && jr < rows;
    if (newrow) {
      if (__any_sync(0xffffffffu, !mbar_wait(&fullv[warp], par))) {
        bad = true;
        break;
      }
      for (int kv = 0; kv < 2; ++kv) {
        const int hs = (kv == 0 ? a.nq : a.nq + a.nkv) + g;  // this KV head's k (or v) among the heads
        __half* dst = reinterpret_cast<__half*>(kv == 0 ? a.kc_w : a.vc_w) + (head_row + pos) * D;
        uint8_t* base = kv == 0 ? ksl : vsl;
        for (int i = lane; i < D; i += 32) {
          const __half hv = __float2half_rn(qkv_at(a, qkv, hs, i, D, pos));
          dst[i] = hv;
          *reinterpret_cast<__half*>(base + (i >> 6) * T::BOX + swz(jr, (i & 63) >> 3) + (i & 7) * 2) = hv;
        }
      }
      __syncwarp();
    }
    // ---- S = Q.K^T: four n-tiles of 8 keys
    float s[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint32_t af[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        const int mi = lane >> 3, key = 8 * (2 * pp + (mi >> 1)) + (lane & 7), chunk = 2 * ks + (mi & 1);
        uint32_t r0, r1, r2, r3;
        ldsm_x4(smem_u32(ksl + (chunk >> 3) * T::BOX + swz(key, chunk & 7)), r0, r1, r2, r3);
        mma16816(s[2 * pp], af, r0, r1);
        mma16816(s[2 * pp + 1], af, r2, r3);
      }
    }
    __syncwarp();
    // the K half is read: copy the next tile's K rows now
    if (lane == 0 && it + 1 < nmine) {
      if (newrow) fence_proxy_async();  // generic stores into the slot before the tensor copy over them
      issue(t + kWarps, 0);
      knext = true;
    }
    // ---- online softmax on this lane's row: keys 8n + 2tq + e; the two halves of q add up
    float sc[4][2];
    float mx = -INFINITY;
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float v = s[n][e] + __shfl_xor_sync(0xffffffffu, s[n][e], XR);
        sc[n][e] = 8 * n + 2 * tq + e < rows ? v : -INFINITY;
        mx = fmaxf(mx, sc[n][e]);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m_run, mx);
    const float al = expf(m_run - mn);  // m_run = -inf on the first tile: 0 (o is 0 anyway)
    float ps = 0.f;
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[n][e] = expf(sc[n][e] - mn);
        ps += sc[n][e];
      }
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    l_run = l_run * al + ps;
    m_run = mn;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      o[n][0] *= al;
      o[n][1] *= al;
    }
    // A fragments of P: k-step kk covers keys 16kk .. 16kk + 15 (n-tiles 2kk, 2kk + 1)
    uint32_t pa[2][2];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t hi = 0u, lo = 0u;
        if (live) split_half2(sc[2 * kk + hf][0], sc[2 * kk + hf][1], hi, lo);
        pa[kk][hf] = rem ? lo : hi;
      }
    // ---- the V half: stale rows past the tile's end are zeroed (P is 0 there, but 0 x NaN is NaN)
    if (!newrow && __any_sync(0xffffffffu, !mbar_wait(&fullv[warp], par))) {
      bad = true;
      break;
    }
    if (rows < TK) {
      for (int i = lane; i < (TK - rows) * T::NB * 8; i += 32) {
        const int r = rows + i / (T::NB * 8), bx = (i / 8) % T::NB, c = i & 7;
        *reinterpret_cast<uint4*>(vsl + bx * T::BOX + r * 128 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }
    // ---- O += P.V: two k-steps of 16 keys, n-tiles of 8 dims in pairs
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t af[4] = {pa[kk][0], 0u, pa[kk][1], 0u};
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        const int mi = lane >> 3, key = 16 * kk + 8 * (mi & 1) + (lane & 7), chunk = 2 * np + (mi >> 1);
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(smem_u32(vsl + (chunk >> 3) * T::BOX + swz(key, chunk & 7)), r0, r1, r2, r3);
        mma16816(o[2 * np], af, r0, r1);
        mma16816(o[2 * np + 1], af, r2, r3);
      }
    }
    __syncwarp();
    if (lane == 0 && it + 1 < nmine) {
      if (newrow || rows < TK) fence_proxy_async();
      issue(t + kWarps, 1);
    }
  }
  if (bad && lane == 0) {
    atomicOr(a.guard, GUARD_TIMEOUT);
    // the copies that may still be in flight into this slot, bounded (as in the scalar kernel)
    const uint32_t par = static_cast<uint32_t>(it) & 1u;
    if (it < nmine) {
      if (!kdone) (void)mbar_wait(&fullk[warp], par);
      if (knext) (void)mbar_wait(&fullk[warp], par ^ 1u);
      (void)mbar_wait(&fullv[warp], par);
    }
  }
  __syncwarp();

  // ---- this warp's (m, l, o) per head into its idle slot: o = fp16 row + remainder row
  float* wst = reinterpret_cast<float*>(ksl);
  if (live && !rem && tq == 0) {
    wst[hq] = m_run;
    wst[REP + hq] = l_run;
  }
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float v = o[n][e] + __shfl_xor_sync(0xffffffffu, o[n][e], XR);
      if (live && !rem) wst[2 * REP + hq * D + 8 * n + 2 * tq + e] = v;
    }
  __syncthreads();
  for (int idx = tid; idx < REP * D; idx += kAttnThreads) {
    const int h = idx / D;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, reinterpret_cast<const float*>(smem + w * T::SLOT)[h]);
    float O = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float* ws = reinterpret_cast<const float*>(smem + w * T::SLOT);
      if (ws[h] != -INFINITY) O = fmaf(ws[2 * REP + idx], expf(ws[h] - M), O);
    }
    cpart[2 * REP + idx] = O;
  }
  if (tid < REP) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, reinterpret_cast<const float*>(smem + w * T::SLOT)[tid]);
    float Ls = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float* ws = reinterpret_cast<const float*>(smem + w * T::SLOT);
      if (ws[tid] != -INFINITY) Ls = fmaf(ws[REP + tid], expf(ws[tid] - M), Ls);
    }
    cpart[tid] = M;
    cpart[REP + tid] = Ls;
  }

  // ---- merge of the cluster's splits through distributed shared memory
  cluster_sync_all();
  const int rank = static_cast<int>(cluster_rank());
  const int chunk = (REP * D + ns - 1) / ns;
  const int lo = rank * chunk, hi = min(REP * D, lo + chunk);
  for (int idx = lo + tid; idx < hi; idx += kAttnThreads) {
    const int h = idx / D;
    float M = -INFINITY;
    for (int s2 = 0; s2 < ns; ++s2) M = fmaxf(M, ld_peer(peer_addr(&cpart[h], s2)));
    float Ls = 0.f, O = 0.f;
    for (int s2 = 0; s2 < ns; ++s2) {
      const float ms = ld_peer(peer_addr(&cpart[h], s2));
      const float w = ms == -INFINITY ? 0.f : expf(ms - M);
      Ls = fmaf(ld_peer(peer_addr(&cpart[REP + h], s2)), w, Ls);
      O = fmaf(ld_peer(peer_addr(&cpart[2 * REP + idx], s2)), w, O);
    }
    store_out(a, static_cast<size_t>(b) * a.nq * D + (g * REP + h) * D + (idx - h * D), O / Ls);
  }
  cluster_sync_all();  // peers read this CTA's cpart until here
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

template <typename K>
cudaError_t attr_one(K kernel, int bytes) {
  cudaError_t e = set_kernel_smem(kernel, bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int D, int REP>
cudaError_t attr_dr(int bytes) {
  cudaError_t e;
  if ((e = attr_one(attn_decode_kernel<D, REP, float>, bytes))) return e;
  if ((e = attr_one(attn_decode_kernel<D, REP, __half>, bytes))) return e;
  if ((e = attr_one(attn_decode_kernel<D, REP, int8_t>, bytes))) return e;
  if constexpr (D % 64 == 0) return attr_one(attn_decode_tc_kernel<D, REP>, bytes + 1024);
  return cudaSuccess;
}

template <int D, int REP>
const void* kernel_ptr(int kv_dtype) {
  switch (kv_dtype) {
    case 0: return reinterpret_cast<const void*>(attn_decode_kernel<D, REP, float>);
    case 2:
      if constexpr (D % 64 == 0) return reinterpret_cast<const void*>(attn_decode_tc_kernel<D, REP>);
      return reinterpret_cast<const void*>(attn_decode_kernel<D, REP, __half>);
    case 3: return reinterpret_cast<const void*>(attn_decode_kernel<D, REP, int8_t>);
  }
  return nullptr;
}

template <int D, int REP>
cudaError_t launch_tc(const AttnArgs& a, const cudaLaunchConfig_t& cfg) {
  if constexpr (D % 64 == 0) {
    cudaLaunchConfig_t c2 = cfg;
    c2.dynamicSmemBytes = static_cast<size_t>(TcTile<D>::SLOT) * kWarps + 1024;
    return cudaLaunchKernelEx(&c2, attn_decode_tc_kernel<D, REP>, *static_cast<const CUtensorMap*>(a.map_k),
                              *static_cast<const CUtensorMap*>(a.map_v), a);
  }
  return cudaErrorInvalidValue;
}

#define K2_ATTN_SHAPES(X) \
  X(16, 1) X(16, 2) X(16, 4) X(64, 1) X(64, 2) X(64, 4) X(128, 1) X(128, 2) X(128, 4)

constexpr size_t kAttnMaxDyn = 200 * 1024;

}  // namespace

bool attn_tc_supported(int head_dim, int rep) {
  return (head_dim == 64 || head_dim == 128) && (rep == 1 || rep == 2 || rep == 4);
}

size_t attn_slot_bytes(int head_dim, int kv_dtype) {
  const size_t elt = kv_dtype == 0 ? 4 : (kv_dtype == 2 ? 2 : 1);
  return 2 * kAttnTK * head_dim * elt + (kv_dtype == 3 ? 2 * kAttnTK * 2 : 0);
}

bool attn_supported(int head_dim, int rep, int kv_dtype) {
  if (kv_dtype != 0 && kv_dtype != 2 && kv_dtype != 3) return false;
  if (attn_slot_bytes(head_dim, kv_dtype) * kWarps > kAttnMaxDyn) return false;
#define K2_ATTN_SUP(D, R) \
  if (head_dim == D && rep == R) return true;
  K2_ATTN_SHAPES(K2_ATTN_SUP)
#undef K2_ATTN_SUP
  return false;
}

cudaError_t attn_init_attrs() {
  cudaError_t e = cudaSuccess;
#define K2_ATTN_ATTR(D, R) \
  if (e == cudaSuccess) e = attr_dr<D, R>(static_cast<int>(kAttnMaxDyn));
  K2_ATTN_SHAPES(K2_ATTN_ATTR)
#undef K2_ATTN_ATTR
  return e;
}

int attn_ctas_per_sm(int head_dim, int rep, int kv_dtype) {
  const void* fn = nullptr;
#define K2_ATTN_PTR(D, R) \
  if (head_dim == D && rep == R) fn = kernel_ptr<D, R>(kv_dtype);
  K2_ATTN_SHAPES(K2_ATTN_PTR)
#undef K2_ATTN_PTR
  int n = 0;
  const size_t dyn = attn_slot_bytes(head_dim, kv_dtype) * kWarps + (kv_dtype == 2 && attn_tc_supported(head_dim, rep) ? 1024 : 0);
  if (!fn || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kAttnThreads, dyn) != cudaSuccess) return 1;
  return n < 1 ? 1 : n;
}

int attn_max_cluster(int head_dim, int rep, int kv_dtype, int limit) {
  const void* fn = nullptr;
#define K2_ATTN_PTR(D, R) \
  if (head_dim == D && rep == R) fn = kernel_ptr<D, R>(kv_dtype);
  K2_ATTN_SHAPES(K2_ATTN_PTR)
#undef K2_ATTN_PTR
  if (!fn) return 0;
  for (int c = limit; c >= 1; --c) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c, 1, 1);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes =
        attn_slot_bytes(head_dim, kv_dtype) * kWarps + (kv_dtype == 2 && attn_tc_supported(head_dim, rep) ? 1024 : 0);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) == cudaSuccess && n >= 1) return c;
    (void)cudaGetLastError();
  }
  return 0;
}

cudaError_t launch_attn(const AttnArgs& a, int head_dim, int rep, int kv_dtype, int nsplit, int batch,
                        cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nsplit, a.nkv, batch);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(a.slot_bytes) * kWarps;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  const bool tc = kv_dtype == 2 && a.map_k != nullptr && a.map_v != nullptr && attn_tc_supported(head_dim, rep);
#define K2_ATTN_LAUNCH(D, R) \
  if (head_dim == D && rep == R) return tc ? launch_tc<D, R>(a, cfg) : launch_dr<D, R>(a, kv_dtype, cfg);
  K2_ATTN_SHAPES(K2_ATTN_LAUNCH)
#undef K2_ATTN_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace k2
