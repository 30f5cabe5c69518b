// Tensor-core GEMM for prefill: D[rows x tokens] = W[rows x K] . X[tokens x K]^T
// on the 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM).
//
// Prefill runs the decoder over a block of T prompt tokens at once (k2-burn
// README, "Status: v0": prefill then single-token decode), so its projections
// are dense contractions.  W is a packed projection matrix (pairs of rows in
// 512-byte chunks, the same copy the decode step streams); a 4-D TMA tensor
// map (element, row-in-pair, chunk, pair) reads it as ordinary 128-row K-major
// tiles.  The operands are one of:
//  - single fp16 (the default prefill, f16 = 1): W the fp16 copy of the bf16
//    weights, X single fp16 activations; one MMA per K step;
//  - bf16 W and X as two bf16 matrices whose sum is the fp32 activation
//    (x_hi = bf16(x), x_lo = bf16(x - x_hi)), one MMA per half, so the product
//    keeps ~16 mantissa bits of the activation; without the low half (LO =
//    false) one MMA on x_hi alone;
//  - with a second weight map (WL = true: W = w_hi + w_lo, the int4 weights
//    dequantized to two bf16 halves) each K step also issues w_lo . x_hi
//    (w_lo . x_lo, below both halves' rounding, is left out).
//
// Two kernels.  tc_gemm_sk_kernel (the prefill's and the batched decode's):
// one persistent CTA per SM; warp 0 issues the TMA loads into a ring, thread
// 32 the MMAs into one of two TMEM accumulators, warps 2-5 drain the other and
// apply the epilogue (store, residual add, SwiGLU), over whole tiles or
// stream-K shares (below).  tc_gemm_kernel: one CTA per 128-row x 128-token
// tile, the epilogue after its own K steps (option K2_OPT_PREFILL_GEMM = 0).
// Every wait is bounded; a timeout sets the guard word and skips the
// accumulator.
#include <cuda.h>

#include <algorithm>

#include "k2_kernels.h"
#include "k2_common.cuh"

namespace k2 {

namespace {

constexpr int BM = 128, BK = 64;
// tile shapes: 128 tokens for prefill, 16 for a batched decode step
// KPS_: K steps per ring stage.  A TMA copy group is taken in by an SM at a
// rate that grows with the bytes requested together (measured: one 16 KB box
// ~69 GB/s, two ~121, four ~142 from L2), not with the number of stages in
// flight, so the prefill kernels (128-token tiles) fill each stage with two K
// steps (one barrier, twice the boxes).
template <int BN_, bool LO_ = true, bool WL_ = false, int KPS_ = 1>
struct Tile {
  static constexpr int BN = BN_;
  static constexpr bool LO = LO_;  // the activations' low half is a second B operand
  static constexpr bool WL = WL_;  // the weights' low half is a second A operand
  static constexpr int KPS = KPS_;
  static constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
  static constexpr int OFF_AL = A_BYTES;                       // one K step: A, [A lo], B, [B lo]
  static constexpr int OFF_B = (WL_ ? 2 : 1) * A_BYTES;
  static constexpr int OFF_BL = OFF_B + B_BYTES;
  static constexpr int STEP_BYTES = OFF_B + (LO_ ? 2 : 1) * B_BYTES;
  static constexpr int STAGE_BYTES = KPS_ * STEP_BYTES;
  static constexpr int STAGES = BN_ >= 128 ? (192 * 1024) / STAGE_BYTES : 8;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;  // + alignment of the ring to 1024 B
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;             // allocation: a power of two >= 32
  // instruction descriptor of kind::f16: bf16 A and B, fp32 D, both K-major
  static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                    (static_cast<uint32_t>(BM >> 4) << 24);
  static_assert(STEP_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "stages stay 1024-byte aligned");
  static_assert(STAGES >= 2, "a ring of at least two stages");
};

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* m, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(m), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_4d(void* dst, const CUtensorMap* m, int c0, int c1, int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(smem_u32(dst)),
      "l"(m), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}
// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row core
// groups 1024 B apart (the layout a 128-byte-swizzled TMA box leaves)
__device__ __forceinline__ uint64_t smem_desc(const void* p) {
  const uint64_t addr = (smem_u32(p) & 0x3FFFFu) >> 4;
  return addr | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// the tile of the non-persistent kernel: two K steps per stage where both fit twice
template <int BN, bool LO, bool WL>
using TileG = Tile<BN, LO, WL, (BN >= 128 && !WL) ? 2 : 1>;

// the instruction descriptor with fp16 A and B (a.f16) instead of bf16: the
// A / B type fields (bits 7-9, 10-12) are 0 for fp16, 1 for bf16
__device__ __forceinline__ uint32_t idesc_for(uint32_t bf16_desc, int f16) {
  return f16 ? (bf16_desc & ~((7u << 7) | (7u << 10))) : bf16_desc;
}
// SwiGLU of one (gate, up) pair into output o: bf16 hi (+ lo), or single fp16 (f16)
__device__ __forceinline__ void swiglu_store(const TcGemmArgs& a, size_t o, float g, float u) {
  const float y = g * __frcp_rn(1.0f + __expf(-g)) * u;
  if (a.f16) {
    if (!(fabsf(y) <= 65504.f)) atomicOr(a.guard, GUARD_RANGE);
    reinterpret_cast<__half*>(a.out_hi)[o] = __float2half_rn(y);
    return;
  }
  __nv_bfloat16 hi = __float2bfloat16_rn(y);
  a.out_hi[o] = hi;
  if (a.out_lo != nullptr) a.out_lo[o] = __float2bfloat16_rn(y - __bfloat162float(hi));
}
__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

template <int BN_, bool LO, bool WL>
__global__ void __launch_bounds__(128, 1) tc_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                                                         const __grid_constant__ CUtensorMap tmWl,
                                                         const __grid_constant__ CUtensorMap tmXh,
                                                         const __grid_constant__ CUtensorMap tmXl, const TcGemmArgs a) {
  using C = TileG<BN_, LO, WL>;
  constexpr int BN = C::BN, STAGES = C::STAGES, KPS = C::KPS;
  constexpr int STAGE_BYTES = C::STAGE_BYTES, STEP_BYTES = C::STEP_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], done;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;  // first token
  const int m0 = blockIdx.y * BM;  // first (packed) weight row
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = tmem_slot;
  // this CTA's K steps (split-K over blockIdx.z)
  const int kb = static_cast<int>((static_cast<long long>(a.ksteps) * blockIdx.z) / a.splits);
  const int ke = static_cast<int>((static_cast<long long>(a.ksteps) * (blockIdx.z + 1)) / a.splits);
  const int nk = ke - kb;
  const int nf = (nk + KPS - 1) / KPS;  // stage fills: KPS K steps each, the last one maybe fewer
  if (threadIdx.x == 0) {  // TMA producer
    int f = 0;
    for (; f < nf; ++f) {
      const int s = f % STAGES;
      if (f >= STAGES && !mbar_wait(&empty[s], static_cast<uint32_t>((f / STAGES) - 1) & 1u)) {
        atomicOr(a.guard, GUARD_TIMEOUT);
        break;
      }
      const int cnt = min(KPS, nk - f * KPS);
      mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(cnt * STEP_BYTES));
      for (int q = 0; q < cnt; ++q) {
        uint8_t* st = smem + s * STAGE_BYTES + q * STEP_BYTES;
        const int kk = (kb + f * KPS + q) * BK;
        tma_4d(st, &tmW, kk & 255, 0, kk >> 8, m0 >> 1, &full[s]);
        if constexpr (WL) tma_4d(st + C::OFF_AL, &tmWl, kk & 255, 0, kk >> 8, m0 >> 1, &full[s]);
        tma_2d(st + C::OFF_B, &tmXh, kk, n0, &full[s]);
        if constexpr (LO) tma_2d(st + C::OFF_BL, &tmXl, kk, n0, &full[s]);
      }
    }
    // copies still in flight must land before the CTA ends: wait for the
    // last ones the MMA thread may not have consumed (bounded)
    for (int j = max(0, f - STAGES); j < f; ++j) mbar_wait(&full[j % STAGES], static_cast<uint32_t>(j / STAGES) & 1u);
  } else if (threadIdx.x == 32) {  // MMA issuer
    for (int f = 0; f < nf; ++f) {
      const int s = f % STAGES;
      if (!mbar_wait(&full[s], static_cast<uint32_t>(f / STAGES) & 1u)) {
        atomicOr(a.guard, GUARD_TIMEOUT);
        break;
      }
      tc_after();
      const int cnt = min(KPS, nk - f * KPS);
      const uint32_t idesc = idesc_for(C::IDESC, a.f16);
      for (int q = 0; q < cnt; ++q) {
        uint8_t* st = smem + s * STAGE_BYTES + q * STEP_BYTES;
#pragma unroll
        for (int j = 0; j < BK / 16; ++j) {
          const uint64_t ad = smem_desc(st + j * 32), bd = smem_desc(st + C::OFF_B + j * 32);
          mma(tmem, ad, bd, idesc, (f | q | j) != 0);
          if constexpr (LO) mma(tmem, ad, smem_desc(st + C::OFF_BL + j * 32), idesc, 1u);
          if constexpr (WL) mma(tmem, smem_desc(st + C::OFF_AL + j * 32), bd, idesc, 1u);
        }
      }
      mma_commit(&empty[s]);
    }
    mma_commit(&done);  // with no K step at all it completes at once
  }
  __syncwarp();
  const bool ok = mbar_wait(&done, 0);
  tc_after();
  if (ok && nk > 0 && (__ldcg(a.guard) & GUARD_TIMEOUT) == 0u) {
    const int row = m0 + warp * 32 + lane;
    const float rs = (a.row_scale != nullptr && row < a.N) ? __ldg(a.row_scale + row) : 1.f;
    constexpr int CW = BN < 32 ? BN : 32;  // accumulator columns read per tcgen05.ld
#pragma unroll 1
    for (int c = 0; c < BN; c += CW) {
      uint32_t v[CW];
      if constexpr (CW == 32) tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, v);
      else tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, v);
#pragma unroll
      for (int j = 0; j < CW; ++j) {
        const int t = n0 + c + j;
        const float acc = a.row_scale != nullptr ? __uint_as_float(v[j]) * rs : __uint_as_float(v[j]);
        if (a.mode == TC_SWIGLU) {  // rows (2p, 2p+1) = (gate_p, up_p): adjacent lanes
          const float up = __shfl_xor_sync(0xffffffffu, acc, 1);
          if (!(lane & 1) && t < a.T && row < a.N) swiglu_store(a, static_cast<size_t>(t) * a.ldo + (row >> 1), acc, up);
        } else if (t < a.T && row < a.N) {
          float* o = a.out + static_cast<size_t>(t) * a.ldo + row;
          if (a.splits > 1) atomicAdd(o, acc);  // partial sums of a split K (the STORE target is zeroed)
          else if (a.mode == TC_RESID) *o += acc;
          else *o = acc;
        }
      }
    }
  } else if (threadIdx.x == 64 && !ok) {
    atomicOr(a.guard, GUARD_TIMEOUT);
  }
  tc_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
}

// a position in a persistent CTA's work: tile, and fill k of it; after the
// tile's last fill the next tile is `step` further on
struct Cursor {
  int tile, k, fpt, step;
  __device__ __forceinline__ void next() {
    if (++k == fpt) {
      k = 0;
      tile += step;
    }
  }
};

// Persistent variant: one CTA per SM, warp 0 loads, warp 1 issues the MMAs
// into one of two TMEM accumulators, warps 2-5 drain the other (warp w reads
// TMEM lanes 32 (w % 4) ..), so accumulation and write-back overlap.  The work
// is a sequence of ring fills of KPS K steps each, over (row tile, token tile)
// pairs ordered tokens-fastest, in one of two shares:
//  - stream-K (a.whole == 0; few row tiles: o_proj, down, the batched decode):
//    an equal share of all (tile, fill) pairs per CTA, so every SM streams the
//    same number of weight bytes; a tile cut by a share boundary is finished
//    with fp32 atomicAdd from both sides (TC_RESID adds to the residual,
//    TC_STORE expects a zeroed target);
//  - whole tiles (a.whole == 1; many tiles: the prefill's QKV and gate/up):
//    CTA b takes tiles b, b + grid, b + 2 grid, ... (at any moment the CTAs
//    share a few weight row tiles and all token tiles in L2), and the
//    epilogue of one tile -- a plain store, the residual add or SwiGLU --
//    runs while the next tile's K steps stream in.
template <int BN_, bool LO, bool WL, int KPS>
__global__ void __launch_bounds__(192, 1) tc_gemm_sk_kernel(const __grid_constant__ CUtensorMap tmW,
                                                            const __grid_constant__ CUtensorMap tmWl,
                                                            const __grid_constant__ CUtensorMap tmXh,
                                                            const __grid_constant__ CUtensorMap tmXl,
                                                            const TcGemmArgs a) {
  using C = Tile<BN_, LO, WL, KPS>;
  constexpr int BN = C::BN, STAGES = C::STAGES, STAGE_BYTES = C::STAGE_BYTES, STEP_BYTES = C::STEP_BYTES;
  constexpr int COLS = C::TMEM_COLS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], accf[2], acce[2];
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tok_tiles = (a.T + BN - 1) / BN;
  const int row_tiles = (2 * ((a.N + 1) / 2) + BM - 1) / BM;
  const int fpt = a.ksteps / KPS;  // ring fills per tile (ksteps is a multiple of 4)
  const int tiles = row_tiles * tok_tiles;
  // this CTA's fills i = 0 .. cnt - 1, walked by a cursor (tile, fill k)
  // that each role advances itself (no division in the loops)
  int cnt = 0;
  Cursor first{0, 0, fpt, 1};
  if (a.whole) {
    cnt = tiles > static_cast<int>(blockIdx.x) ? ((tiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1) * fpt : 0;
    first = Cursor{static_cast<int>(blockIdx.x), 0, fpt, static_cast<int>(gridDim.x)};
  } else {
    const long long total = static_cast<long long>(tiles) * fpt;
    const long long g0 = total * blockIdx.x / gridDim.x;
    cnt = static_cast<int>(total * (blockIdx.x + 1) / gridDim.x - g0);
    first = Cursor{static_cast<int>(g0 / fpt), static_cast<int>(g0 % fpt), fpt, 1};
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);  // one arrival per epilogue warp
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(2 * COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = tmem_slot;
  if (threadIdx.x == 0) {  // TMA producer
    // the fill at cursor c into stage memory st: its weight and / or activation boxes
    auto load = [&](uint8_t* st, const Cursor& c, bool w, bool x, uint64_t* bar) {
      const int rt = c.tile / tok_tiles;
      const int m0 = rt * BM, n0 = (c.tile - rt * tok_tiles) * BN;
#pragma unroll
      for (int q = 0; q < KPS; ++q) {
        uint8_t* sq = st + q * STEP_BYTES;
        const int kk = (c.k * KPS + q) * BK;
        if (w) {
          tma_4d(sq, &tmW, kk & 255, 0, kk >> 8, m0 >> 1, bar);
          if constexpr (WL) tma_4d(sq + C::OFF_AL, &tmWl, kk & 255, 0, kk >> 8, m0 >> 1, bar);
        }
        if (x) {
          tma_2d(sq + C::OFF_B, &tmXh, kk, n0, bar);
          if constexpr (LO) tma_2d(sq + C::OFF_BL, &tmXl, kk, n0, bar);
        }
      }
    };
    // Under programmatic dependent launch the weights of the first stages are
    // requested before waiting for the previous kernel (they never depend on
    // it); the activations of those stages follow once it has completed.
    const int pre = min(STAGES, cnt);
    Cursor c = first;
    for (int j = 0; j < pre; ++j, c.next()) {
      mbar_arrive_expect_tx(&full[j], STAGE_BYTES);
      load(smem + j * STAGE_BYTES, c, true, false, &full[j]);
    }
    pdl_wait();
    pdl_trigger();
    c = first;
    for (int j = 0; j < pre; ++j, c.next()) load(smem + j * STAGE_BYTES, c, false, true, &full[j]);
    int i = pre, s = pre % STAGES;
    uint32_t ph = pre / STAGES;  // how often the ring wrapped before fill i
    for (; i < cnt; ++i, c.next()) {
      if (i >= STAGES && !mbar_wait(&empty[s], (ph - 1) & 1u)) {
        atomicOr(a.guard, GUARD_TIMEOUT);
        break;
      }
      mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
      load(smem + s * STAGE_BYTES, c, true, true, &full[s]);
      if (++s == STAGES) {
        s = 0;
        ++ph;
      }
    }
    for (int j = max(0, i - STAGES); j < i; ++j) mbar_wait(&full[j % STAGES], static_cast<uint32_t>(j / STAGES) & 1u);
  } else if (threadIdx.x == 32) {  // MMA issuer
    int piece = 0, s = 0, k = first.k;
    uint32_t ph = 0;
    bool start = true;  // the first fill of a piece: the accumulator is overwritten
    for (int i = 0; i < cnt; ++i) {
      const int b = piece & 1;
      if (start && piece >= 2 && !mbar_wait(&acce[b], static_cast<uint32_t>((piece >> 1) - 1) & 1u)) {
        atomicOr(a.guard, GUARD_TIMEOUT);
        break;
      }
      if (!mbar_wait(&full[s], ph & 1u)) {
        atomicOr(a.guard, GUARD_TIMEOUT);
        break;
      }
      tc_after();
      const uint32_t acc = tmem + b * COLS;
      const uint32_t idesc = idesc_for(C::IDESC, a.f16);
#pragma unroll
      for (int q = 0; q < KPS; ++q) {
        uint8_t* st = smem + s * STAGE_BYTES + q * STEP_BYTES;
#pragma unroll
        for (int j = 0; j < BK / 16; ++j) {
          const uint64_t ad = smem_desc(st + j * 32), bd = smem_desc(st + C::OFF_B + j * 32);
          mma(acc, ad, bd, idesc, (!start || q != 0 || j != 0) ? 1u : 0u);
          if constexpr (LO) mma(acc, ad, smem_desc(st + C::OFF_BL + j * 32), idesc, 1u);
          if constexpr (WL) mma(acc, smem_desc(st + C::OFF_AL + j * 32), bd, idesc, 1u);
        }
      }
      mma_commit(&empty[s]);
      start = false;
      if (k == fpt - 1 || i == cnt - 1) {  // this CTA's piece of the tile ends
        mma_commit(&accf[b]);
        ++piece;
        start = true;
      }
      if (++k == fpt) k = 0;
      if (++s == STAGES) {
        s = 0;
        ++ph;
      }
    }
  } else if (warp >= 2) {  // epilogue: drain each piece's accumulator
    const int lg = (warp & 3) * 32;  // the TMEM lanes (tile rows) this warp may read
    pdl_wait();  // the output (residual or zeroed target) is the previous kernels'
    int piece = 0, i = 0;
    Cursor c = first;
    while (i < cnt) {
      const int len = min(cnt - i, fpt - c.k);  // this piece's fills
      const int tile = c.tile;
      const int b = piece & 1;
      const bool ok = mbar_wait(&accf[b], static_cast<uint32_t>(piece >> 1) & 1u);
      if (__any_sync(0xffffffffu, !ok)) {
        if (lane == 0) atomicOr(a.guard, GUARD_TIMEOUT);
        break;
      }
      tc_after();
      const int rt = tile / tok_tiles;
      const int row = rt * BM + lg + lane;
      const int n0t = (tile - rt * tok_tiles) * BN;
      const float rs = (a.row_scale != nullptr && row < a.N) ? __ldg(a.row_scale + row) : 1.f;
      // the accumulator in parts of at most 128 columns (registers); the
      // buffer is released once its last part is in registers
      constexpr int PART = BN > 128 ? 128 : BN;
#pragma unroll 1
      for (int p0 = 0; p0 < BN; p0 += PART) {
        uint32_t v[PART];
        if constexpr (PART == 16) {
          tmem_ld16(tmem + b * COLS + (static_cast<uint32_t>(lg) << 16) + p0, v);
        } else {
#pragma unroll
          for (int c = 0; c < PART; c += 32)
            tmem_ld32(tmem + b * COLS + (static_cast<uint32_t>(lg) << 16) + p0 + c, v + c);
        }
        if (p0 + PART == BN) {
          tc_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce[b]);
        }
        const int n0 = n0t + p0;
        if (!a.whole) {
          if (row < a.N) {
#pragma unroll
            for (int j = 0; j < PART; ++j)
              if (n0 + j < a.T) atomicAdd(a.out + static_cast<size_t>(n0 + j) * a.ldo + row, __uint_as_float(v[j]) * rs);
          }
        } else if (a.mode == TC_SWIGLU) {
          // rows (2p, 2p+1) = (gate_p, up_p) sit in adjacent lanes; per pair of
          // columns (j, j+1) the even lane finishes column j and the odd lane
          // column j+1, each after one exchange
          const bool odd = lane & 1;
#pragma unroll
          for (int j = 0; j < PART; j += 2) {
            const float a0 = __uint_as_float(v[j]) * rs, a1 = __uint_as_float(v[j + 1]) * rs;
            const float recv = __shfl_xor_sync(0xffffffffu, odd ? a0 : a1, 1);
            const float g = odd ? recv : a0, u = odd ? a1 : recv;
            const int t = n0 + j + (odd ? 1 : 0);
            if (t < a.T && row < a.N) swiglu_store(a, static_cast<size_t>(t) * a.ldo + (row >> 1), g, u);
          }
        } else if (row < a.N) {
#pragma unroll
          for (int j = 0; j < PART; ++j) {
            if (n0 + j < a.T) {
              float* o = a.out + static_cast<size_t>(n0 + j) * a.ldo + row;
              const float y = __uint_as_float(v[j]) * rs;
              if (a.mode == TC_RESID) *o += y;
              else *o = y;
            }
          }
        }
      }
      i += len;
      c.k += len;
      if (c.k == fpt) {
        c.k = 0;
        c.tile += c.step;
      }
      ++piece;
    }
  }
  tc_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * COLS) : "memory");
}

typedef CUresult (*EncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}

// ---- causal prefill attention on the 5th-generation tensor cores -------------------------------
// One CTA takes 128 query rows -- 128 / REP tokens x the REP query heads of one
// KV head -- and walks the cached keys 0 .. (its last position) in tiles of 64:
//   S = Q.K^T   (tcgen05.mma M=128 N=64, S in TMEM): Q as fp16 hi + lo halves
//               (two MMAs per k-step: ~22 bits of every query; SPLIT = false:
//               fp16 Q alone, one MMA), K the fp16 cache;
//   softmax     row r (TMEM lane r) is shared by the NQ warps that may read
//               lane group r / 32 (NQ = 4 for head_dim 128, 2 for 64): each
//               takes 64 / NQ of the tile's 64 scores (tcgen05.ld), they
//               exchange their maxima through shared memory, and write their
//               parts of P = 2^(s - m) as fp16 hi + lo (SPLIT = false: fp16 P
//               alone);
//   O += P.V^T  (tcgen05.mma M=128 N=D, O in TMEM).
// Q, K and P are K-major with the 128-byte swizzle (the layout of the GEMMs'
// descriptors): Q and P are written so by the threads, K arrives so by TMA; V
// enters P.V as it arrives, [key][dim] rows, through an MN-major descriptor
// (dims contiguous: 64-dim swizzle atoms LBO apart, 8-key groups SBO apart).
// The tensor pipe never waits for the softmax: S of the next tile is issued
// (into the other of two S buffers) before this tile's softmax, and P is
// double-buffered, so P.V of one tile overlaps the next one's softmax.  Scores
// are kept in base 2 (Q carries log2(e)), so p = 2^(s - m) is one ex2 each.
// A row's reference maximum only moves when a tile's maximum exceeds it by
// more than kRescaleLog2 (then O and the row's sums are rescaled in TMEM);
// otherwise p may exceed 1 (at most 2^kRescaleLog2, well inside fp16), and the
// final division by the sum makes the result exact anyway.  K/V tiles rotate
// through STAGES stages (4 with single-operand Q and P, 3 with hi + lo): tile
// kt + STAGES - 2 is requested once the P.V that read the stage it reuses (of
// tile kt - 2) is done, so each copy has STAGES - 2 softmax passes to land.
// 4 NQ softmax warps (NQ per TMEM lane group) and one issuer warp
constexpr int kPaRows = 128, kPaKeys = 64, kPaMaxSoftWarps = 16;
constexpr float kRescaleLog2 = 11.0f;
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float ex2(float x) {  // 2^x (the SFU's approximation; 2^-inf = 0)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, bool SPLIT>
struct PaSmem {
  // softmax warps per TMEM lane group (4, a quarter row each, measured slower:
  // 4096-token prefill 52.4 against 50.3 ms)
  static constexpr int NQ = 2;
  static constexpr int SOFT = 4 * NQ, THREADS = 32 * (SOFT + 1);
  static constexpr int NA = D / 64;                   // 64-dim swizzle atoms per row
  static constexpr int Q = kPaRows * 128;             // one atom of the 128 query rows (16 KB)
  static constexpr int KT = kPaKeys * 128;            // one atom of a 64-key K (or V) tile (8 KB)
  static constexpr int STAGE = 2 * NA * KT;           // K and V of one tile
  static constexpr int P = kPaRows * 128;             // P [128][64 keys] (one half)
  static constexpr int PB = (SPLIT ? 2 : 1) * P;       // one P buffer: hi (+ lo)
  static constexpr int STAGES = SPLIT ? 3 : 4;        // K/V stages (5 measured no faster than 4)
  static constexpr int PD = STAGES - 2;               // tiles requested ahead of the one being scored
  static constexpr int OFF_QH = 0, OFF_QL = OFF_QH + NA * Q;
  static constexpr int OFF_ST = OFF_QL + (SPLIT ? NA * Q : 0);  // STAGES stages
  static constexpr int OFF_P = OFF_ST + STAGES * STAGE;        // two P buffers
  static constexpr int BYTES = OFF_P + 2 * PB;
  static constexpr int DYN = BYTES + 1024;            // + alignment to 1024 B
  static constexpr int TMEM_COLS = D + 128 <= 128 ? 128 : 256;  // O [D], then S [64] x 2
  // instruction descriptors (kind::f16): fp16 A and B, fp32 D, M = 128; S: both K-major;
  // O: B (V) MN-major (bit 16)
  static constexpr uint32_t IDESC_S = (1u << 4) | (static_cast<uint32_t>(kPaKeys >> 3) << 17) | (8u << 24);
  static constexpr uint32_t IDESC_O =
      (1u << 4) | (1u << 16) | (static_cast<uint32_t>(D >> 3) << 17) | (8u << 24);
};

// byte offset of element (row r, column e) in a K-major 128-byte-swizzled block of 64 columns
__device__ __forceinline__ uint32_t sw128(int r, int e) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((((e >> 3) ^ (r & 7)) & 7) << 4) + (e & 7) * 2);
}
// shared-memory matrix descriptor, MN-major with the 128-byte swizzle: rows of
// 128 bytes along K (8-row groups sbo bytes apart), 64-element atoms along MN
// lbo bytes apart
__device__ __forceinline__ uint64_t smem_desc_mn(const void* p, uint32_t lbo, uint32_t sbo) {
  const uint64_t addr = (smem_u32(p) & 0x3FFFFu) >> 4;
  return addr | (static_cast<uint64_t>(lbo >> 4) << 16) | (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* m, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(dst)),
      "l"(m), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <int D, int REP, bool SPLIT>
__global__ void __launch_bounds__(PaSmem<D, SPLIT>::THREADS, 1) prefill_attn_tc_kernel(const __grid_constant__ KvMaps maps,
                                                                        const PrefillAttnArgs a) {
  using Sm = PaSmem<D, SPLIT>;
  constexpr int NA = Sm::NA;
  constexpr int QT = kPaRows / REP;  // tokens per CTA
  constexpr int NQ = Sm::NQ, kPaSoftWarps = Sm::SOFT, kPaStages = Sm::STAGES;
  constexpr int CW = kPaKeys / NQ;   // score columns per thread and tile
  constexpr int DH = D / NQ;         // O columns per thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[kPaStages], sbar[2], obar[2], sfree[2], pready[2];
  __shared__ uint32_t tmem_slot;
  __shared__ float xmax[NQ][kPaRows];    // each part's tile maximum per row
  __shared__ int pbad[kPaMaxSoftWarps];  // a softmax warp's verdict, read by the warps sharing its rows
  __shared__ int issued[3];            // the issuer's count of K/V tiles, S and P.V issued
  // the GEMM that reads this kernel's output may launch at once and request its
  // weights on SMs this grid leaves idle (it waits for this grid before reading)
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = (warp & 3) * 32 + lane;  // TMEM lane = query row
  const int hf = warp >> 2;                // which CW of the 64 scores (and DH columns of O) this thread takes
  // the last query blocks (the most keys) are scheduled first, so the final
  // wave holds the short ones
  const int t0 = (gridDim.x - 1 - blockIdx.x) * QT, g = blockIdx.y;
  const int nt = min(QT, a.n - t0);
  const int tq = row / REP, hh = row - tq * REP;  // token t0 + tq, query head g * REP + hh
  const bool row_ok = tq < nt;
  const int qpos = a.pos0 + t0 + tq;              // the row's position: it sees keys 0 .. qpos
  const int kend = a.pos0 + t0 + nt;              // keys of the CTA: 0 .. kend - 1
  const int nkt = (kend + kPaKeys - 1) / kPaKeys;
  const int krow0 = a.head_row0 + g * a.cap;      // tensor row of key 0 of this KV head

  if (tid == 0) {
    for (int st = 0; st < kPaStages; ++st) mbar_init(&full[st], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sbar[b], 1);
      mbar_init(&obar[b], 1);
      mbar_init(&sfree[b], kPaSoftWarps);
      mbar_init(&pready[b], kPaSoftWarps);
    }
    fence_mbar_init();
  }
  if (tid < kPaSoftWarps) pbad[tid] = 0;
  if (tid < 3) issued[tid] = 0;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(Sm::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // this row's half of Q (pre-scaled by 1 / sqrt(D)) as fp16 hi + lo, swizzled
  if (warp < kPaSoftWarps) {
    const float* q = a.Q + static_cast<size_t>(t0 + tq) * a.nq * D + (g * REP + hh) * D;
#pragma unroll
    for (int cc = 0; cc < D / (8 * NQ); ++cc) {
      const int c = hf * (D / (8 * NQ)) + cc;  // 8-dim chunk
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = row_ok ? q[8 * c + e] * (a.scale * kLog2e) : 0.f;  // base-2 scores
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split_half2(v[2 * e], v[2 * e + 1], hi[e], lo[e]);
      const uint32_t off = (c >> 3) * Sm::Q + sw128(row, 8 * (c & 7));
      *reinterpret_cast<uint4*>(smem + Sm::OFF_QH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      if constexpr (SPLIT) *reinterpret_cast<uint4*>(smem + Sm::OFF_QL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
  fence_proxy_async();  // generic stores (Q) before the MMAs read them
  auto issue_tile = [&](int kt) {
    const int st = kt % kPaStages;
    uint8_t* base = smem + Sm::OFF_ST + st * Sm::STAGE;
    mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(Sm::STAGE));
#pragma unroll
    for (int at = 0; at < NA; ++at) {
      tma_3d(base + at * Sm::KT, &maps.k, 64 * at, krow0 + kt * kPaKeys, a.layer, &full[st]);
      tma_3d(base + (NA + at) * Sm::KT, &maps.v, 64 * at, krow0 + kt * kPaKeys, a.layer, &full[st]);
    }
  };
  const bool issuer = tid == kPaSoftWarps * 32;  // lane 0 of the last warp issues every copy and MMA
  tc_before();
  __syncthreads();  // the barriers (initialised by thread 0) and Q are ready
  tc_after();
  if (issuer)
    for (int kt = 0; kt <= Sm::PD && kt < nkt; ++kt) issue_tile(kt);
  const uint32_t tmem = tmem_slot;
  // thread 0: S of tile kt = Q.K^T into S buffer kt & 1 (hi and lo halves of Q)
  auto issue_s = [&](int kt) {
    const uint8_t* kst = smem + Sm::OFF_ST + (kt % kPaStages) * Sm::STAGE;
    const uint32_t ts = tmem + D + 64 * (kt & 1);
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      const uint64_t kd = smem_desc(kst + (j >> 2) * Sm::KT + (j & 3) * 32);
      mma(ts, smem_desc(smem + Sm::OFF_QH + (j >> 2) * Sm::Q + (j & 3) * 32), kd, Sm::IDESC_S, j > 0 ? 1u : 0u);
      if constexpr (SPLIT) mma(ts, smem_desc(smem + Sm::OFF_QL + (j >> 2) * Sm::Q + (j & 3) * 32), kd, Sm::IDESC_S, 1u);
    }
    mma_commit(&sbar[kt & 1]);
  };
  // the issuer: P.V of tile kt (hi and lo halves of P) into O, V straight from its stage
  auto issue_pv = [&](int kt) {
    const int b = kt & 1;
    const uint8_t* ph = smem + Sm::OFF_P + b * Sm::PB;
    const uint8_t* vst = smem + Sm::OFF_ST + (kt % kPaStages) * Sm::STAGE + NA * Sm::KT;
#pragma unroll
    for (int j = 0; j < kPaKeys / 16; ++j) {
      const uint64_t vd = smem_desc_mn(vst + j * 16 * 128, Sm::KT, 8 * 128);  // keys 16j .. 16j + 15
      mma(tmem, smem_desc(ph + j * 32), vd, Sm::IDESC_O, (kt > 0 || j > 0) ? 1u : 0u);
      if constexpr (SPLIT) mma(tmem, smem_desc(ph + Sm::P + j * 32), vd, Sm::IDESC_O, 1u);
    }
    mma_commit(&obar[b]);
  };
  const uint32_t lanes = static_cast<uint32_t>((warp & 3) * 32) << 16;  // this warp's TMEM lanes
  const uint32_t t_o = tmem + lanes + hf * DH;                             // this thread's part of O

  float m_ref = -INFINITY, l_part = 0.f;  // the row's reference maximum; this half's sum of p
  bool bad = false;
  if (warp == kPaSoftWarps) {
    // The issuer: S of tile kt once its K/V stage has landed and its S buffer
    // has been read (tile kt - 2); then P.V of tile kt - 1 once all softmax
    // warps have written its P, and the copy of tile kt + PD into the stage of
    // tile kt - 2 once that tile's P.V is done.  The softmax warps never wait
    // for one another.
    if (issuer) {
      int t_is = min(nkt, Sm::PD + 1), s_is = 0, o_is = 0;
      for (int kt = 0; kt < nkt && !bad; ++kt) {
        const int b = kt & 1;
        if (!mbar_wait(&full[kt % kPaStages], static_cast<uint32_t>(kt / kPaStages) & 1u) ||
            (kt >= 2 && !mbar_wait(&sfree[b], static_cast<uint32_t>((kt - 2) >> 1) & 1u))) {
          bad = true;
          break;
        }
        tc_after();
        issue_s(kt);
        s_is = kt + 1;
        if (kt >= 1) {
          if (!mbar_wait(&pready[(kt - 1) & 1], static_cast<uint32_t>((kt - 1) >> 1) & 1u)) {
            bad = true;
            break;
          }
          tc_after();
          issue_pv(kt - 1);
          o_is = kt;
          if (kt + Sm::PD < nkt) {
            if (kt >= 2 && !mbar_wait(&obar[b], static_cast<uint32_t>((kt - 2) >> 1) & 1u)) {
              bad = true;
              break;
            }
            issue_tile(kt + Sm::PD);
            t_is = kt + Sm::PD + 1;
          }
        }
      }
      if (!bad && nkt > 0) {
        if (mbar_wait(&pready[(nkt - 1) & 1], static_cast<uint32_t>((nkt - 1) >> 1) & 1u)) {
          tc_after();
          issue_pv(nkt - 1);
          o_is = nkt;
        } else {
          bad = true;
        }
      }
      issued[0] = t_is;
      issued[1] = s_is;
      issued[2] = o_is;
    }
  } else {
    for (int kt = 0; kt < nkt; ++kt) {
      const int b = kt & 1;
      // the P.V of two tiles ago, which read P buffer b, is done
      if (kt >= 2 && !mbar_wait(&obar[b], static_cast<uint32_t>((kt - 2) >> 1) & 1u)) bad = true;
      // the CTA's last tile: V rows past its last key (stale cache rows, maybe
      // not even finite) become zeros, since P.V multiplies them by p = 0
      const int kvalid = kend - kt * kPaKeys;
      if (kvalid < kPaKeys) {
        if (!mbar_wait(&full[kt % kPaStages], static_cast<uint32_t>(kt / kPaStages) & 1u)) bad = true;
        if (!__any_sync(0xffffffffu, bad)) {
          uint8_t* vst = smem + Sm::OFF_ST + (kt % kPaStages) * Sm::STAGE + NA * Sm::KT;
          const int chunks = (kPaKeys - kvalid) * 8;  // 16-byte chunks per 64-dim atom
          for (int i = tid; i < NA * chunks; i += 32 * kPaSoftWarps) {
            const int at = i / chunks, r = i - at * chunks;
            *reinterpret_cast<uint4*>(vst + at * Sm::KT + (kvalid + r / 8) * 128 + (r & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      bad = __any_sync(0xffffffffu, bad);
      // this thread's 32 scores of the row; then the S buffer is free for tile kt + 2
      if (!mbar_wait(&sbar[b], static_cast<uint32_t>(kt >> 1) & 1u)) bad = true;
      bad = __any_sync(0xffffffffu, bad);
      tc_after();
      float sv[CW];
      if (!bad) {
        uint32_t raw[CW];
        if constexpr (CW == 32) tmem_ld32(tmem + lanes + D + 64 * b + CW * hf, raw);
        else tmem_ld16(tmem + lanes + D + 64 * b + CW * hf, raw);
#pragma unroll
        for (int j = 0; j < CW; ++j) sv[j] = __uint_as_float(raw[j]);
      } else {
#pragma unroll
        for (int j = 0; j < CW; ++j) sv[j] = -INFINITY;
      }
      tc_before();
      __syncwarp();
      if (lane == 0 && !bad) mbar_arrive(&sfree[b]);
      float mx = -INFINITY;
      const int last = row_ok ? qpos - kt * kPaKeys - CW * hf : -1;  // this part's last visible column
      if (__any_sync(0xffffffffu, last < CW - 1)) {  // a column to mask in this warp's rows
#pragma unroll
        for (int j = 0; j < CW; ++j) sv[j] = j <= last ? sv[j] : -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < CW; ++j) mx = fmaxf(mx, sv[j]);
      // the row's other parts are taken by warps w + 4q: a barrier of those NQ
      // warps, which also share their verdicts, so all of them leave together
      xmax[hf][row] = mx;
      if (lane == 0) pbad[warp] = bad ? 1 : 0;
      asm volatile("bar.sync %0, %1;" ::"r"(1 + (warp & 3)), "r"(32 * NQ) : "memory");
      float mt = mx;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (pbad[(warp & 3) + 4 * q] != 0) bad = true;
        mt = fmaxf(mt, xmax[q][row]);
      }
      asm volatile("bar.sync %0, %1;" ::"r"(1 + (warp & 3)), "r"(32 * NQ) : "memory");  // xmax / pbad reused next tile
      if (bad) break;
      // the reference maximum moves only when a tile's maximum exceeds it by kRescaleLog2
      const bool move = row_ok && mt > -INFINITY && (m_ref == -INFINITY || mt > m_ref + kRescaleLog2);
      const float alpha = move ? (m_ref == -INFINITY ? 0.f : ex2(m_ref - mt)) : 1.f;
      if (move) {
        l_part *= alpha;
        m_ref = mt;
      }
      if (kt > 0 && __any_sync(0xffffffffu, move)) {  // this half of O *= alpha (a warp-wide access)
        // every earlier P.V must be done: the one of the previous tile may still run
        const bool ok = mbar_wait(&obar[b ^ 1], static_cast<uint32_t>((kt - 1) >> 1) & 1u);
        if (__any_sync(0xffffffffu, !ok)) {
          // the partner warp learns it at the next tile's exchange, where both
          // leave (leaving here could strand it at that barrier)
          bad = true;
          continue;
        }
        tc_after();
        uint32_t ov[32];
#pragma unroll 1
        for (int c = 0; c < DH; c += 32) {
          tmem_ld32(t_o + c, ov);
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
          tmem_st32(t_o + c, ov);
        }
      }
      // P = 2^(s - m_ref) as fp16 hi + lo, this part's CW keys
      {
        uint8_t* ph = smem + Sm::OFF_P + b * Sm::PB;
        uint8_t* pl = ph + Sm::P;
        const float mr = m_ref == -INFINITY ? 0.f : m_ref;  // a row with no visible key yet: all p are 0
        float ps = 0.f;
#pragma unroll
        for (int c = 0; c < CW / 8; ++c) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            // masked columns are -inf: 2^-inf = 0
            const float p0 = ex2(sv[8 * c + 2 * e] - mr), p1 = ex2(sv[8 * c + 2 * e + 1] - mr);
            ps += p0 + p1;
            split_half2(p0, p1, hi[e], lo[e]);
          }
          const uint32_t off = sw128(row, CW * hf + 8 * c);
          *reinterpret_cast<uint4*>(ph + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          if constexpr (SPLIT) *reinterpret_cast<uint4*>(pl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        l_part += ps;
      }
      fence_proxy_async();  // P and the zeroed V rows (generic stores) before the MMAs read them
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pready[b]);
    }
  }
  bad = __syncthreads_or(bad) != 0;  // one verdict for the CTA
  const int t_issued = issued[0], s_issued = issued[1], o_issued = issued[2];
  // copies and MMAs still in flight end before the CTA's memory goes away (bounded waits)
  if (bad && issuer) {
    atomicOr(a.guard, GUARD_TIMEOUT);
    for (int k = max(0, t_issued - kPaStages); k < t_issued; ++k)
      (void)mbar_wait(&full[k % kPaStages], static_cast<uint32_t>(k / kPaStages) & 1u);
    if (s_issued > 0) (void)mbar_wait(&sbar[(s_issued - 1) & 1], static_cast<uint32_t>((s_issued - 1) >> 1) & 1u);
  }
  bool have_o = o_issued > 0;
  for (int k = max(0, o_issued - 2); k < o_issued; ++k)
    if (!mbar_wait(&obar[k & 1], static_cast<uint32_t>(k >> 1) & 1u)) have_o = false;
  have_o = __syncthreads_and(have_o) != 0;  // the tensor-memory reads below are warp-wide
  tc_after();
  // the row's sum: all its parts (softmax warps only)
  float l_sum = 0.f;
  if (warp < kPaSoftWarps) {
    xmax[hf][row] = l_part;
    asm volatile("bar.sync %0, %1;" ::"r"(1 + (warp & 3)), "r"(32 * NQ) : "memory");
#pragma unroll
    for (int q = 0; q < NQ; ++q) l_sum += xmax[q][row];
  }
  if (warp < kPaSoftWarps && !bad && have_o) {
    // this part of the row: O / sum, as bf16 hi (+ lo when the GEMM that follows takes it), or fp16
    const float inv = l_sum > 0.f ? 1.0f / l_sum : 0.f;
    const size_t ob = static_cast<size_t>(t0 + tq) * a.nq * D + (g * REP + hh) * D + hf * DH;
#pragma unroll 1
    for (int c = 0; c < DH; c += 32) {
      uint32_t ov[32];
      tmem_ld32(t_o + c, ov);
      if (row_ok && a.f16out) {  // single fp16 (attention outputs are averages of V rows: inside its range)
#pragma unroll
        for (int j = 0; j < 32; j += 2)
          *reinterpret_cast<__half2*>(reinterpret_cast<__half*>(a.oh) + ob + c + j) =
              __floats2half2_rn(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv);
      } else if (row_ok) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          __nv_bfloat16 h0, l0, h1, l1;
          split_bf16(__uint_as_float(ov[j]) * inv, h0, l0);
          split_bf16(__uint_as_float(ov[j + 1]) * inv, h1, l1);
          *reinterpret_cast<__nv_bfloat162*>(a.oh + ob + c + j) = __nv_bfloat162(h0, h1);
          if (a.ol != nullptr) *reinterpret_cast<__nv_bfloat162*>(a.ol + ob + c + j) = __nv_bfloat162(l0, l1);
        }
      }
    }
  } else if (issuer && !bad && o_issued > 0 && !have_o) {
    atomicOr(a.guard, GUARD_TIMEOUT);
  }
  tc_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Sm::TMEM_COLS) : "memory");
}

}  // namespace

bool tc_encode_weight(void* map, const void* packed, int N, int K) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const int CT = (K + 255) / 256, npairs = (N + 1) / 2;
  cuuint64_t dims[4] = {256, 2, static_cast<cuuint64_t>(CT), static_cast<cuuint64_t>(npairs)};
  cuuint64_t strides[3] = {512, 1024, static_cast<cuuint64_t>(CT) * 1024};
  cuuint32_t box[4] = {BK, 2, 1, BM / 2}, es[4] = {1, 1, 1, 1};
  return enc(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(packed), dims,
             strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_encode_act(void* map, const void* buf, int rows, int K, int tile_tokens) {
  EncodeTiled enc = encode_fn();
  if (!enc || K % 8 != 0 || (tile_tokens != 16 && tile_tokens != 128 && tile_tokens != 256)) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {BK, static_cast<cuuint32_t>(tile_tokens)}, es[2] = {1, 1};
  return enc(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(buf), dims,
             strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One layer's K or V cache as a 2-D tensor [rows][head_dim] of fp16, read by
// the tensor-core decode attention in boxes of 64 dims x 32 rows with the
// 128-byte swizzle (the layout its ldmatrix fragments expect).
bool attn_encode_kv(void* map, const void* base, long long rows, int head_dim) {
  EncodeTiled enc = encode_fn();
  if (!enc || head_dim % 64 != 0 || rows <= 0) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kAttnTK)}, es[2] = {1, 1};
  return enc(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
             strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool attn_encode_kv_layers(void* map, const void* base, long long rows, int head_dim, int layers,
                           unsigned long long layer_stride, int box_rows) {
  EncodeTiled enc = encode_fn();
  if (!enc || head_dim % 64 != 0 || rows <= 0 || layers <= 0 || layer_stride % 16 != 0 || box_rows < 1 ||
      box_rows > 256)
    return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(layers)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2, layer_stride};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1}, es[3] = {1, 1, 1};
  return enc(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims,
             strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool prefill_attn_tc_supported(int head_dim, int rep) { return (head_dim == 64 || head_dim == 128) && rep == 4; }

cudaError_t prefill_attn_tc_init_attrs() {
  const auto set = [](const void* k, int bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  };
  cudaError_t e = set(reinterpret_cast<const void*>(prefill_attn_tc_kernel<128, 4, true>), PaSmem<128, true>::DYN);
  if (e == cudaSuccess) e = set(reinterpret_cast<const void*>(prefill_attn_tc_kernel<128, 4, false>), PaSmem<128, false>::DYN);
  if (e == cudaSuccess) e = set(reinterpret_cast<const void*>(prefill_attn_tc_kernel<64, 4, true>), PaSmem<64, true>::DYN);
  if (e == cudaSuccess) e = set(reinterpret_cast<const void*>(prefill_attn_tc_kernel<64, 4, false>), PaSmem<64, false>::DYN);
  return e;
}

cudaError_t launch_prefill_attn_tc(const KvMaps& maps, const PrefillAttnArgs& a, int head_dim, int rep,
                                   cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  if (!prefill_attn_tc_supported(head_dim, rep) || (a.split && a.ol == nullptr)) return cudaErrorInvalidValue;
  const dim3 grid((a.n + kPaRows / rep - 1) / (kPaRows / rep), a.nkv);
  if (head_dim == 128 && a.split)
    prefill_attn_tc_kernel<128, 4, true><<<grid, PaSmem<128, true>::THREADS, PaSmem<128, true>::DYN, s>>>(maps, a);
  else if (head_dim == 128)
    prefill_attn_tc_kernel<128, 4, false><<<grid, PaSmem<128, false>::THREADS, PaSmem<128, false>::DYN, s>>>(maps, a);
  else if (a.split)
    prefill_attn_tc_kernel<64, 4, true><<<grid, PaSmem<64, true>::THREADS, PaSmem<64, true>::DYN, s>>>(maps, a);
  else
    prefill_attn_tc_kernel<64, 4, false><<<grid, PaSmem<64, false>::THREADS, PaSmem<64, false>::DYN, s>>>(maps, a);
  return cudaGetLastError();
}

template <typename K>
cudaError_t smem_attr(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t tc_gemm_init_attrs() {
  cudaError_t e = smem_attr(tc_gemm_kernel<128, true, false>, TileG<128, true, false>::SMEM_BYTES);
  if (e == cudaSuccess) e = smem_attr(tc_gemm_kernel<128, false, false>, TileG<128, false, false>::SMEM_BYTES);
  if (e == cudaSuccess) e = smem_attr(tc_gemm_kernel<128, true, true>, TileG<128, true, true>::SMEM_BYTES);
  if (e == cudaSuccess) e = smem_attr(tc_gemm_kernel<16, true, false>, TileG<16, true, false>::SMEM_BYTES);
  if (e == cudaSuccess) e = smem_attr(tc_gemm_sk_kernel<16, true, false, 1>, Tile<16, true, false, 1>::SMEM_BYTES);
  if (e == cudaSuccess) e = smem_attr(tc_gemm_sk_kernel<128, true, false, 1>, Tile<128, true, false, 1>::SMEM_BYTES);
  if (e == cudaSuccess) e = smem_attr(tc_gemm_sk_kernel<128, false, false, 1>, Tile<128, false, false, 1>::SMEM_BYTES);
  if (e == cudaSuccess) e = smem_attr(tc_gemm_sk_kernel<128, true, true, 1>, Tile<128, true, true, 1>::SMEM_BYTES);
  if (e == cudaSuccess) e = smem_attr(tc_gemm_sk_kernel<128, true, false, 2>, Tile<128, true, false, 2>::SMEM_BYTES);
  if (e == cudaSuccess) e = smem_attr(tc_gemm_sk_kernel<128, false, false, 2>, Tile<128, false, false, 2>::SMEM_BYTES);
  if (e == cudaSuccess) e = smem_attr(tc_gemm_sk_kernel<256, false, false, 1>, Tile<256, false, false, 1>::SMEM_BYTES);
  return e;
}

cudaError_t launch_tc_gemm_sk(const void* mapW, const void* mapWl, const void* mapXh, const void* mapXl,
                              const TcGemmArgs& a, int ctas, cudaStream_t s, bool pdl) {
  if (a.T <= 0) return cudaSuccess;
  if ((a.tile_tokens != 16 && a.tile_tokens != 128 && a.tile_tokens != 256) || (a.mode == TC_SWIGLU && !a.whole) ||
      ctas < 1 || a.ksteps % 4 != 0)
    return cudaErrorInvalidValue;
  const int tt = a.tile_tokens;
  const bool lo = mapXl != nullptr, wl = mapWl != nullptr;
  if ((tt == 16 && (!lo || wl)) || (wl && !lo) || (tt == 256 && (lo || wl))) return cudaErrorInvalidValue;
  // 128-token tiles fill each ring stage with two K steps (larger copy groups: measured on the
  // 4096-token prefill, 85.0 -> 80.2 ms with the stream-K o_proj / down so too) where two fit
  // twice; 256-token tiles take one K step (48 KB) per stage, four stages (49.5 -> 48.8 ms)
  const bool two = tt == 128 && !wl;
  const long long tiles = static_cast<long long>((2 * ((a.N + 1) / 2) + BM - 1) / BM) * ((a.T + tt - 1) / tt);
  const int grid = static_cast<int>(std::min<long long>(ctas, a.whole ? tiles : tiles * a.ksteps));
  const CUtensorMap& w = *static_cast<const CUtensorMap*>(mapW);
  const CUtensorMap& wlo = *static_cast<const CUtensorMap*>(wl ? mapWl : mapW);  // unread without it
  const CUtensorMap& xh = *static_cast<const CUtensorMap*>(mapXh);
  const CUtensorMap& xl = *static_cast<const CUtensorMap*>(lo ? mapXl : mapXh);  // unread without the low half
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = tt == 16    ? Tile<16, true, false, 1>::SMEM_BYTES
                         : tt == 256 ? Tile<256, false, false, 1>::SMEM_BYTES
                         : wl        ? Tile<128, true, true, 1>::SMEM_BYTES
                         : two    ? (lo ? Tile<128, true, false, 2>::SMEM_BYTES : Tile<128, false, false, 2>::SMEM_BYTES)
                         : lo     ? Tile<128, true, false, 1>::SMEM_BYTES
                                  : Tile<128, false, false, 1>::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (tt == 16) return cudaLaunchKernelEx(&cfg, tc_gemm_sk_kernel<16, true, false, 1>, w, wlo, xh, xl, a);
  if (tt == 256) return cudaLaunchKernelEx(&cfg, tc_gemm_sk_kernel<256, false, false, 1>, w, wlo, xh, xl, a);
  if (wl) return cudaLaunchKernelEx(&cfg, tc_gemm_sk_kernel<128, true, true, 1>, w, wlo, xh, xl, a);
  if (two && lo) return cudaLaunchKernelEx(&cfg, tc_gemm_sk_kernel<128, true, false, 2>, w, wlo, xh, xl, a);
  if (two) return cudaLaunchKernelEx(&cfg, tc_gemm_sk_kernel<128, false, false, 2>, w, wlo, xh, xl, a);
  if (lo) return cudaLaunchKernelEx(&cfg, tc_gemm_sk_kernel<128, true, false, 1>, w, wlo, xh, xl, a);
  return cudaLaunchKernelEx(&cfg, tc_gemm_sk_kernel<128, false, false, 1>, w, wlo, xh, xl, a);
}

cudaError_t launch_tc_gemm(const void* mapW, const void* mapWl, const void* mapXh, const void* mapXl,
                           const TcGemmArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.splits < 1 || (a.splits > 1 && a.mode == TC_SWIGLU)) return cudaErrorInvalidValue;
  const bool lo = mapXl != nullptr, wl = mapWl != nullptr;
  if (wl && (!lo || a.tile_tokens != 128)) return cudaErrorInvalidValue;
  const CUtensorMap& w = *static_cast<const CUtensorMap*>(mapW);
  const CUtensorMap& wlo = *static_cast<const CUtensorMap*>(wl ? mapWl : mapW);  // unread without it
  const CUtensorMap& xh = *static_cast<const CUtensorMap*>(mapXh);
  const CUtensorMap& xl = *static_cast<const CUtensorMap*>(lo ? mapXl : mapXh);  // unread without the low half
  const int rows = (2 * ((a.N + 1) / 2) + BM - 1) / BM;
  const dim3 g16((a.T + 15) / 16, rows, a.splits), g128((a.T + 127) / 128, rows, a.splits);
  if (a.tile_tokens == 16 && lo && !wl) {
    tc_gemm_kernel<16, true, false><<<g16, 128, TileG<16, true, false>::SMEM_BYTES, s>>>(w, wlo, xh, xl, a);
  } else if (a.tile_tokens == 128 && wl) {
    tc_gemm_kernel<128, true, true><<<g128, 128, TileG<128, true, true>::SMEM_BYTES, s>>>(w, wlo, xh, xl, a);
  } else if (a.tile_tokens == 128 && lo) {
    tc_gemm_kernel<128, true, false><<<g128, 128, TileG<128, true, false>::SMEM_BYTES, s>>>(w, wlo, xh, xl, a);
  } else if (a.tile_tokens == 128) {
    tc_gemm_kernel<128, false, false><<<g128, 128, TileG<128, false, false>::SMEM_BYTES, s>>>(w, wlo, xh, xl, a);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace k2
