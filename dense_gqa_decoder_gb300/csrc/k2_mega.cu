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
// all SMs once.
//
// Streaming: the weights and cached K/V rows never depend on the
// activations, so each warp streams them continuously: its producer lane
// walks one fixed sequence of 10 KB slots spanning every phase of the step
// (its share of the QKV weights, then its K/V tiles, then its o_proj,
// gate/up, down weights, then the next layer's ...) and refills a ring slot
// as soon as it is consumed.  Each refill is one bulk copy (cp.async.bulk,
// mbarrier complete_tx) of a contiguous run of the packed weights (pairs of
// rows in 512-byte chunks) or of one K/V tile.
//
// Synchronisation is dataflow, not grid barriers: every activation element
// is stored as one 64-bit word (fp32 value, 32-bit tag) with a relaxed
// gpu-scope store, the tag naming the launch and the phase that wrote it.
// A consumer loads the words it needs and retries those whose tag is not yet
// the producer phase's; a 64-bit access is single-copy atomic, so a matching
// tag carries its value.  This folds "wait for the phase" and "load the
// input" into one L2 round trip.  Reuse of a buffer is safe because every
// CTA owns rows of every GEMV output (the grid is never larger than the
// smallest pair count): a CTA can only overwrite a buffer after it has seen
// outputs that every CTA wrote after its last read of that buffer.
//
// Phases of a layer: QKV GEMV (+ GroupedRMSNorm, + split-half RoPE) | GQA
// attention partials per (KV head, key split) with the KV append, merged by
// the last split of each KV head | o_proj GEMV + residual | gate/up GEMV +
// SwiGLU | down GEMV + residual.  Then final norm + lm_head GEMV +
// first-index argmax (kimi-k3-in-c k3_run.c, `argmax_`).  The residual rows
// of a CTA stay in its shared memory from one residual phase to the next.
// Every wait is bounded (GUARD_TIMEOUT).
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
// Packed weight formats: one unit holds a 512-byte chunk of both rows of a
// pair (UNIT bytes; int4: 256 bytes of codes per row and the two rows' 8
// block scales of the chunk); EPL weights per lane and row in a chunk.
template <typename PT>
struct Fmt {
  static constexpr int UNIT = 1024, EPL = Unpack<PT>::N;
};
template <>
struct Fmt<q4_block64> {
  static constexpr int UNIT = kQ4Unit, EPL = kQ4Chunk / 32;
};
static_assert(SB % Fmt<__nv_bfloat16>::UNIT == 0 && SB % Fmt<q4_block64>::UNIT == 0, "slots hold whole units");
constexpr int PX = 10;           // float4 groups of the input vector per thread (K <= 10240)
// keys per attention tile: the K and V rows (plus int8 scales) fit one slot
template <int D, typename KVT>
constexpr int tile_keys() {
  return (2 * kMegaTK * D * static_cast<int>(sizeof(KVT)) + 4 * kMegaTK <= SB) ? kMegaTK
         : (2 * (kMegaTK / 2) * D * static_cast<int>(sizeof(KVT)) + 4 * (kMegaTK / 2) <= SB) ? kMegaTK / 2
                                                                                               : 0;
}
static_assert(2 * MW <= 32, "the warp-split GEMV records fit one warp");
constexpr int kPhases = 5;       // per layer: QKV, ATTN, O, GU, DOWN
enum { PH_QKV = 0, PH_ATTN = 1, PH_O = 2, PH_GU = 3, PH_DOWN = 4 };

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

// ---- tagged activations ----------------------------------------------------------------------
typedef unsigned long long u64;
__device__ __forceinline__ void st_tagged(u64* p, float v, uint32_t tag) {
  const u64 w = (static_cast<u64>(tag) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ void ld_tagged2(const u64* p, u64& w0, u64& w1) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(w0), "=l"(w1) : "l"(p) : "memory");
}
__device__ __forceinline__ u64 ld_tagged(const u64* p) {
  u64 w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}
__device__ __forceinline__ bool tag_is(u64 w, uint32_t tag) { return static_cast<uint32_t>(w >> 32) == tag; }
__device__ __forceinline__ float tag_val(u64 w) { return __uint_as_float(static_cast<uint32_t>(w)); }

// Bounded retry loop: false (and GUARD_TIMEOUT) once the wait has run out.
struct Patience {
  uint64_t limit;
  uint64_t t0 = 0;
  __device__ __forceinline__ explicit Patience(uint64_t limit_ns) : limit(limit_ns) {}
  __device__ __forceinline__ bool more(unsigned* guard) {
    const uint64_t t = globaltimer();
    if (t0 == 0) t0 = t;
    if (t - t0 > limit) {
      atomicOr(guard, GUARD_TIMEOUT);
      return false;
    }
    if (kMegaPollSleepNs > 0) __nanosleep(kMegaPollSleepNs);
    return true;
  }
};

__device__ __forceinline__ unsigned long long sm_clock() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void trace_mark(const MegaArgs& a, int q, int k) {
  if (a.trace != nullptr && threadIdx.x == 0)
    a.trace[(static_cast<size_t>(q) * gridDim.x + blockIdx.x) * 4 + k] = sm_clock();
}

// x[e .. e+3] for e = tid * 4 + i * MT * 4 (i < PX, e < K) from tagged words.
__device__ bool poll_x(const u64* tv, int K, uint32_t tag, float4* xq, unsigned* guard, uint64_t limit_ns) {
  const int tid = threadIdx.x;
  unsigned pend = 0;
#pragma unroll
  for (int i = 0; i < PX; ++i) {
    xq[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid * 4 + i * MT * 4 < K) pend |= 1u << i;
  }
  Patience wait(limit_ns);
  while (pend) {
    u64 w[PX][4];
#pragma unroll
    for (int i = 0; i < PX; ++i) {  // every load first, then the checks
      w[i][0] = w[i][1] = w[i][2] = w[i][3] = 0;
      if (pend & (1u << i)) {
        const u64* p = tv + tid * 4 + i * MT * 4;
        ld_tagged2(p, w[i][0], w[i][1]);
        ld_tagged2(p + 2, w[i][2], w[i][3]);
      }
    }
#pragma unroll
    for (int i = 0; i < PX; ++i) {
      if ((pend & (1u << i)) && tag_is(w[i][0], tag) && tag_is(w[i][1], tag) && tag_is(w[i][2], tag) &&
          tag_is(w[i][3], tag)) {
        xq[i] = make_float4(tag_val(w[i][0]), tag_val(w[i][1]), tag_val(w[i][2]), tag_val(w[i][3]));
        pend &= ~(1u << i);
      }
    }
    if (pend && !wait.more(guard)) return false;
  }
  return true;
}

static_assert(MW * 2 * (kQ4GroupRows / 2) * 2 <= 512, "int4 split-tile records fit the query buffer");
struct MegaShared {
  uint64_t full[MW][NS];
  float ss[MW][4];
  float rs[4];
  int rec_pair[MW][2];
  float rec_val[MW][2][2];
  int rec_n[MW];
  Best best[MW];
  int flag;
  float rsd[2 * kMegaPairsMax];     // this CTA's residual rows, kept from one residual phase to the next
  uint64_t gbar[2];                 // the two norm-gain buffers
  float2 rope_pos[64];              // (cos, sin) at this step's position, i < head_dim / 2
  float qs[512];                    // the query heads of one KV head, scaled (rep * head_dim <= 512)
  int4 wr[5][MW];                   // per GEMV kind: this CTA's pairs [x, y), this warp's units [z, w)
  int4 item;                        // this CTA's attention item: KV head, split, first key, end key
  const void* gains[2 * kMegaMaxLayers + 1];  // attn_norm[l] at 2l, mlp_norm[l] at 2l + 1, final last
  float newkv[2][128];              // the new token's K and V rows (head_dim <= 128)
};

// ---- int4 tiles on the tensor cores -------------------------------------------------
// One mma.sync m16n8k16 (fp16 in, fp32 accumulate) over 16 weights of the 16
// rows of an int4 tile.  A: the lane's tile word w (layout with kWfmtQ4): each
// nibble pair OR-ed into the exponent of fp16 1024 gives 1024 + n (rows g) or
// 1024 + 16 n (rows g + 8) exactly, and one fp16 add or fma turns that into
// the code n - 8, exactly.  B: the input as fp16 high and low halves in
// columns 0 and 1 (lanes 0..7 hold them; the other columns are zero), so D
// column 0 + column 1 is the product with ~22 bits of the input.
__device__ __forceinline__ void q4_tile_mma(uint32_t w, const uint32_t* xf, int lane, float* d) {
  constexpr uint32_t kOne024 = 0x64006400u;  // fp16 1024 in both halves
  const uint32_t w8 = w >> 8;
  uint32_t a[4] = {(w & 0x000F000Fu) | kOne024, (w & 0x00F000F0u) | kOne024, (w8 & 0x000F000Fu) | kOne024,
                   (w8 & 0x00F000F0u) | kOne024};
  const __half2 lo_off = __float2half2_rn(-1032.f), hi_mul = __float2half2_rn(0.0625f),
                hi_off = __float2half2_rn(-72.f);
#pragma unroll
  for (int i = 0; i < 4; i += 2) {
    const __half2 r0 = __hadd2(*reinterpret_cast<const __half2*>(&a[i]), lo_off);
    const __half2 r1 = __hfma2(*reinterpret_cast<const __half2*>(&a[i + 1]), hi_mul, hi_off);
    a[i] = *reinterpret_cast<const uint32_t*>(&r0);
    a[i + 1] = *reinterpret_cast<const uint32_t*>(&r1);
  }
  uint2 b = make_uint2(0u, 0u);
  if (lane < 8) b = *reinterpret_cast<const uint2*>(xf + 2 * lane);
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y));
}

// One mma.sync m16n8k16 over 16 weights of the 16 rows of an fp8 tile: the
// lane's two tile words (layout with kWfmtQ4) hold its 8 E4M3 codes, each pair
// converted to an A fragment register (exact); B as in q4_tile_mma.
__device__ __forceinline__ void f8_tile_mma(uint32_t w0, uint32_t w1, const uint32_t* xf, int lane, float* d) {
  uint32_t a[4];
  const uint32_t w[2] = {w0, w1};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw h =
        __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i >> 1] >> (16 * (i & 1))), __NV_E4M3);
    a[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  uint2 b = make_uint2(0u, 0u);
  if (lane < 8) b = *reinterpret_cast<const uint2*>(xf + 2 * lane);
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y));
}

// ---- static description of the step ------------------------------------------------
// GEMV kinds: 0 QKV, 1 o_proj, 2 gate/up, 3 down, 4 lm_head.  Row ranges do not
// depend on the layer, so they are computed once per launch (shared memory).
struct GDesc {
  const uint8_t* W;
  int N, K, CT, kind;
  const void* gain;
  const float* scale;  // fp8 weights: the row scales (null otherwise)
};

__device__ __forceinline__ GDesc gdesc(const MegaArgs& a, const MegaShared& sh, int q, int qkv_n, int head_dim) {
  GDesc d;
  const int l = q / kPhases, j = q - (q / kPhases) * kPhases;
  if (l >= a.n_layers) {  // the lm_head phase
    d.W = static_cast<const uint8_t*>(a.lm_head); d.N = a.vocab; d.K = a.hidden; d.CT = a.g_lm.CT; d.kind = 4;
    d.gain = a.final_norm;
    d.scale = a.sc_lm;
    return d;
  }
  const size_t ul = static_cast<size_t>(l);
  auto lsc = [&](const float* base, size_t stride) { return base ? base + ul * stride : nullptr; };
  if (j == PH_QKV) {
    d.W = a.w_qkv + ul * a.ws_qkv; d.N = qkv_n; d.K = a.hidden; d.CT = a.g_qkv.CT; d.kind = 0;
    d.gain = sh.gains[2 * l];
    d.scale = lsc(a.sc_qkv, a.ss_qkv);
  } else if (j == PH_O) {
    d.W = a.w_o + ul * a.ws_o; d.N = a.hidden; d.K = a.nq * head_dim; d.CT = a.g_o.CT; d.kind = 1; d.gain = nullptr;
    d.scale = lsc(a.sc_o, a.ss_o);
  } else if (j == PH_GU) {
    d.W = a.w_gu + ul * a.ws_gu; d.N = 2 * a.inter; d.K = a.hidden; d.CT = a.g_gu.CT; d.kind = 2;
    d.gain = sh.gains[2 * l + 1];
    d.scale = lsc(a.sc_gu, a.ss_gu);
  } else {
    d.W = a.w_down + ul * a.ws_down; d.N = a.hidden; d.K = a.inter; d.CT = a.g_down.CT; d.kind = 3; d.gain = nullptr;
    d.scale = lsc(a.sc_down, a.ss_down);
  }
  return d;
}

struct GRange {
  int p0, p1, ua, ub, nslots;  // the CTA's pairs [p0, p1); the warp's units [ua, ub)
};

// the split of kind k's rows over CTAs and of a CTA's units over warps
__device__ __forceinline__ int4 g_split(int N, int CT, int cta, int G, int warp) {
  const int npairs = (N + 1) / 2;
  const int p0 = static_cast<int>((static_cast<long long>(npairs) * cta) / G);
  const int p1 = static_cast<int>((static_cast<long long>(npairs) * (cta + 1)) / G);
  const long long U = static_cast<long long>(p1 - p0) * CT;
  return make_int4(p0, p1, static_cast<int>((U * warp) / MW), static_cast<int>((U * (warp + 1)) / MW));
}

template <int SU>  // packed units per slot
__device__ __forceinline__ GRange g_range(const GDesc& d, const MegaShared& sh, int warp) {
  const int4 w = sh.wr[d.kind][warp];
  GRange r;
  r.p0 = w.x;
  r.p1 = w.y;
  r.ua = w.z;
  r.ub = w.w;
  r.nslots = (r.ub - r.ua + SU - 1) / SU;
  return r;
}

struct AItem {
  int g, sp, k0, k1, ntile;
};

// keys [k0, k1) of split sp of L keys (k0 a multiple of 8: 16-byte int8-scale copies)
__device__ __forceinline__ int4 a_split(const MegaArgs& a, int item, int L) {
  const int ns = a.nsplit;
  const int g = item / ns, sp = item - (item / ns) * ns;
  const int k0 = min(L, static_cast<int>((static_cast<long long>(L) * sp) / ns) & ~7);
  const int k1 = (sp == ns - 1) ? L : min(L, static_cast<int>((static_cast<long long>(L) * (sp + 1)) / ns) & ~7);
  return make_int4(g, sp, k0, k1);
}

template <int TKM>
__device__ __forceinline__ AItem a_item(const MegaShared& sh) {
  AItem it;
  it.g = sh.item.x;
  it.sp = sh.item.y;
  it.k0 = sh.item.z;
  it.k1 = sh.item.w;
  it.ntile = it.k1 > it.k0 ? (it.k1 - it.k0 + TKM - 1) / TKM : 0;
  return it;
}

template <int TKM>
__device__ __forceinline__ int a_mine(const AItem& it, int warp) {
  return it.ntile > warp ? (it.ntile - warp + MW - 1) / MW : 0;
}

// fp16 caches with head_dim a multiple of 64: the attention phase runs on the
// tensor cores, its K/V tiles copied by TMA tensor copies (128-byte swizzle)
template <int D, typename KVT>
constexpr bool tc_attn() {
  return std::is_same<KVT, __half>::value && D % 64 == 0;
}
// a swizzled attention box: kMegaTK rows of 128 bytes (64 fp16 dims)
constexpr int kTcBox = kMegaTK * 128;
// byte offset of 16-byte chunk c (0..7) of row r inside a box (128-byte swizzle)
__device__ __forceinline__ uint32_t swz128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}
__device__ __forceinline__ void tma_3d_hint(void* dst, const CUtensorMap* m, int c0, int c1, int c2, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(m), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ---- the per-warp stream of slots (state kept in lane 0) -----------------------------------
// The producer lane walks every phase q = layer * kPhases + j (then the lm_head
// phase) in order; enter() caches where the current phase's copies come from.
template <int UB, int D, typename KVT>  // UB: bytes of a packed weight unit
struct Stream {
  static constexpr int SU = SB / UB;  // packed units per slot
  static constexpr int TKM = tile_keys<D, KVT>();
  static constexpr int ROWB = D * sizeof(KVT);
  static constexpr bool I8 = std::is_same<KVT, int8_t>::value;
  static constexpr bool TC = tc_attn<D, KVT>();
  int q = 0, k = 0, n = 0, issued = 0, lastq = 0;
  bool done = false, attn = false;
  const uint8_t* src = nullptr;  // GEMV: next unit to copy
  int left = 0;                  // GEMV: units still to copy
  const uint8_t* kb = nullptr;   // attention: K / V rows and scales of this KV head
  const uint8_t* vb = nullptr;
  const __half* ksb = nullptr;
  const __half* vsb = nullptr;
  int j0 = 0, k1 = 0;
  uint64_t policy = 0;  // L2 evict-first: weights and K/V history are read once per step
  const MegaShared* shp = nullptr;
  const KvMaps* maps = nullptr;  // TC: the tensor maps of the caches
  int trow = 0, tlay = 0;        // TC: the tensor row of key 0 of this KV head, the layer

  __device__ void enter(const MegaArgs& a, int cta, int G, int warp, int pos, int qkv_n) {
    k = 0;
    n = 0;
    attn = false;
    if (q > lastq) return;
    const int l = q / kPhases, j = q - (q / kPhases) * kPhases;
    if (l < a.n_layers && j == PH_ATTN) {
      if (cta >= a.nkv * a.nsplit) return;
      const AItem it = a_item<TKM>(*shp);
      const size_t head_row = (static_cast<size_t>(a.seq) * a.nkv + it.g) * a.cap;
      attn = true;
      n = a_mine<TKM>(it, warp);
      kb = a.kc + static_cast<size_t>(l) * a.s_kv + head_row * ROWB;
      vb = a.vc + static_cast<size_t>(l) * a.s_kv + head_row * ROWB;
      if constexpr (I8) {
        ksb = reinterpret_cast<const __half*>(a.ks + static_cast<size_t>(l) * a.s_sc) + head_row;
        vsb = reinterpret_cast<const __half*>(a.vs + static_cast<size_t>(l) * a.s_sc) + head_row;
      }
      j0 = it.k0 + warp * TKM;
      k1 = it.k1;
      trow = static_cast<int>(head_row);
      tlay = l;
      return;
    }
    const GDesc d = gdesc(a, *shp, q, qkv_n, D);
    const GRange r = g_range<SU>(d, *shp, warp);
    n = r.nslots;
    src = d.W + (static_cast<size_t>(r.p0) * d.CT + r.ua) * UB;
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

  __device__ void start(const MegaArgs& a, const MegaShared& sh, const KvMaps* km, uint8_t* ring, uint64_t* full,
                        int cta, int G, int warp, int pos, int qkv_n) {
    shp = &sh;
    maps = km;
    lastq = a.n_layers * kPhases - 1 + (a.head ? 1 : 0);
    policy = l2_evict_first_policy();
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
    if (attn && TC) {
      // whole boxes of kMegaTK rows (rows past the tile are masked by the consumer)
      constexpr int NB = D / 64;
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(2 * NB * kTcBox));
#pragma unroll
      for (int bx = 0; bx < NB; ++bx) {
        tma_3d_hint(dst + bx * kTcBox, &maps->k, 64 * bx, trow + j0, tlay, bar, policy);
        tma_3d_hint(dst + (NB + bx) * kTcBox, &maps->v, 64 * bx, trow + j0, tlay, bar, policy);
      }
      j0 += MW * TKM;
    } else if (attn) {
      const int rows = min(TKM, k1 - j0);
      const int crow = max(0, min(rows, pos - j0));  // cached rows; row pos is written this step
      const int srow = (crow + 7) & ~7;
      const uint32_t bytes = 2u * crow * ROWB + (I8 && crow > 0 ? 2u * srow * 2u : 0u);
      if (bytes == 0) {
        mbar_arrive(bar);
      } else {
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s_hint(dst, kb + static_cast<size_t>(j0) * ROWB, crow * ROWB, bar, policy);
        bulk_g2s_hint(dst + TKM * ROWB, vb + static_cast<size_t>(j0) * ROWB, crow * ROWB, bar, policy);
        if constexpr (I8) {
          bulk_g2s(dst + 2 * TKM * ROWB, ksb + j0, srow * 2u, bar);
          bulk_g2s(dst + 2 * TKM * ROWB + TKM * 2, vsb + j0, srow * 2u, bar);
        }
      }
      j0 += MW * TKM;
    } else {
      const int nu = min(SU, left);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nu) * UB);
      bulk_g2s_hint(dst, src, static_cast<uint32_t>(nu) * UB, bar, policy);
      src += static_cast<size_t>(nu) * UB;
      left -= nu;
    }
    ++issued;
    if (++k >= n) {
      n = 0;
      next_phase(a, cta, G, warp, pos, qkv_n);
    }
  }

  // what issue_next would copy next, asked of L2 instead (on a copy of the
  // stream: the real one is not advanced)
  __device__ void prefetch_next(const MegaArgs& a, int cta, int G, int warp, int pos, int qkv_n) {
    if (done) return;
    if (attn) {
      const int rows = min(TKM, k1 - j0);
      const int crow = max(0, min(rows, pos - j0));
      if (crow > 0) {
        bulk_prefetch_l2(kb + static_cast<size_t>(j0) * ROWB, crow * ROWB);
        bulk_prefetch_l2(vb + static_cast<size_t>(j0) * ROWB, crow * ROWB);
      }
      j0 += MW * TKM;
    } else {
      const int nu = min(SU, left);
      bulk_prefetch_l2(src, static_cast<uint32_t>(nu) * UB);
      src += static_cast<size_t>(nu) * UB;
      left -= nu;
    }
    ++issued;
    if (++k >= n) {
      n = 0;
      next_phase(a, cta, G, warp, pos, qkv_n);
    }
  }
};

// The next `count` slots of a warp's stream beyond those in flight, fetched
// into L2 (called by the producer lane once per phase, off the hot loop).
template <int UB, int D, typename KVT>
__device__ __noinline__ void stream_prefetch(Stream<UB, D, KVT> s, const MegaArgs& a, int cta, int G, int warp,
                                             int pos, int qkv_n, int count) {
  for (int i = 0; i < count && !s.done; ++i) s.prefetch_next(a, cta, G, warp, pos, qkv_n);
}

// The norm gains reach shared memory by bulk copies issued one gain phase
// ahead (a DRAM read under the full weight stream waits several
// microseconds): gain phase number `used` reads buffer used & 1.
struct GainQ {
  int used = 0;    // gain phases entered
  int issued = 0;  // gain copies issued (thread 0)
};
__device__ __forceinline__ uint8_t* gain_buf(uint8_t* smem, int b) {
  return smem + kMegaRingBytes + kMegaXBytes + b * kMegaGainBytes;
}
// the gain of the first gain phase after phase q (null if none)
__device__ __forceinline__ const void* next_gain(const MegaArgs& a, const MegaShared& sh, int q) {
  const int l = q / kPhases, j = q - (q / kPhases) * kPhases;
  if (l >= a.n_layers) return nullptr;
  if (j < PH_GU) return sh.gains[2 * l + 1];
  if (l + 1 < a.n_layers) return sh.gains[2 * l + 2];
  return a.head ? a.final_norm : nullptr;
}
__device__ __forceinline__ void issue_gain(const MegaArgs& a, uint8_t* smem, MegaShared& sh, GainQ& gq,
                                           const void* g, int bytes) {
  const int b = gq.issued & 1;  // last read (generic loads, completed) two gain phases ago
  mbar_arrive_expect_tx(&sh.gbar[b], static_cast<uint32_t>(bytes));
  bulk_g2s(gain_buf(smem, b), g, static_cast<uint32_t>(bytes), &sh.gbar[b]);
  ++gq.issued;
}

struct GEpi {
  int epi;          // EPI_QKV, EPI_RESID, EPI_SWIGLU or EPI_ARGMAX
  u64* out;         // tagged output
  float* plain;     // RESID: also a plain fp32 copy (the residual leaving the last layer)
  const float2* rope;
  int pos;
  int head_dim;
  int n_rot;
  float* logits;
  unsigned* guard;
  uint32_t tag;     // written with this tag
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
template <typename WT>
__device__ __forceinline__ float4 load4_shared(const WT* p, int e);
template <>
__device__ __forceinline__ float4 load4_shared<__nv_bfloat16>(const __nv_bfloat16* p, int e) {
  const uint2 v = *reinterpret_cast<const uint2*>(p + e);
  return make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
}
template <>
__device__ __forceinline__ float4 load4_shared<float>(const float* p, int e) {
  return *reinterpret_cast<const float4*>(p + e);
}
template <typename WT>
__device__ __forceinline__ float load1(const WT* p, size_t e) {
  return to_f32(p[e]);
}

// One GEMV phase: build x in shared memory (waiting for its tags), then
// consume this warp's slots (already in flight) and refill the ring from the
// stream.  x comes from xt (tagged, written by the previous phase with tag
// tag_in) or, in the first phase, from x0f (fp32) or x0w (an embedding row).
// rsd0f / rsd0w: where the first residual phase takes its old residual rows.
template <typename WT, typename PT, int D, typename KVT>
__device__ bool g_phase(const MegaArgs& a, int q, const GDesc& d, const u64* xt, uint32_t tag_in, const float* x0f,
                        const WT* x0w, const float* rsd0f, const WT* rsd0w, const GEpi& ep, uint8_t* smem,
                        MegaShared& sh, Stream<Fmt<PT>::UNIT, D, KVT>& st, GainQ& gq, int& consumed, Best& best,
                        int cta, int G, int pos, int qkv_n) {
  constexpr bool Q4 = std::is_same<PT, q4_block64>::value;
  constexpr int UNIT = Fmt<PT>::UNIT, SU = SB / UNIT;
  constexpr int EPL = Fmt<PT>::EPL;  // packed weights per lane and row in a 512-byte chunk
  constexpr int CH = 32 * EPL;
  constexpr int NPL = EPL / 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = d.K, CT = d.CT;
  float* xs = reinterpret_cast<float*>(smem + kMegaRingBytes);
  uint8_t* ring = smem + static_cast<size_t>(warp) * NS * SB;
  const GRange r = g_range<SU>(d, sh, warp);
  // fp8 / int4 gate/up and lm_head: r.p0 / r.p1 count 16-row tiles (8 pairs
  // each); P0 / P1 are pairs
  constexpr bool F8 = std::is_same<PT, __nv_fp8_e4m3>::value;
  const bool tiles = (Q4 || F8) && tiled_kind(d.kind);
  const int npairs = (d.N + 1) / 2;
  const int P0 = tiles ? r.p0 * (kQ4GroupRows / 2) : r.p0;
  const int P1 = tiles ? min(r.p1 * (kQ4GroupRows / 2), npairs) : r.p1;
  if (lane == 0) sh.rec_n[warp] = 0;

  // ---- x, normalised if the phase has a gain, lane-interleaved per chunk
  bool bad = false;
  {
    const int KP = tiles ? CT * kQ4Block : CT * CH;  // <= PX * MT * 4
    const int gsz = d.gain ? K / a.groups : K;
    auto xidx = [&](int e) {
      const int c = e / CH, rr = e - c * CH, l = rr / EPL, j = rr - l * EPL;
      return ((c * NPL + j / 4) * 32 + l) * 4;
    };
    // a gain phase: its gain was copied one gain phase ago; start the next one
    const WT* gsm = nullptr;
    int gb = 0, guse = 0;
    if (d.gain != nullptr) {
      gb = gq.used & 1;
      guse = gq.used >> 1;
      gsm = reinterpret_cast<const WT*>(gain_buf(smem, gb));
      ++gq.used;
      const void* ng = next_gain(a, sh, q);
      if (tid == 0 && ng != nullptr) issue_gain(a, smem, sh, gq, ng, K * static_cast<int>(sizeof(WT)));
    }
    float side = 0.f;
    const int nrows = min(2 * P1, d.N) - 2 * P0;
    if (ep.epi == EPI_RESID && (rsd0f || rsd0w) && tid < nrows)
      side = rsd0f ? __ldcg(rsd0f + 2 * P0 + tid) : load1(rsd0w, 2 * P0 + tid);
    float4 xq[PX];
    if (xt) {
      bad = !poll_x(xt, K, tag_in, xq, a.guard, a.poll_limit_ns);
    } else {
#pragma unroll
      for (int i = 0; i < PX; ++i) {
        const int e = tid * 4 + i * MT * 4;
        xq[i] = e >= K ? make_float4(0.f, 0.f, 0.f, 0.f)
                       : (x0f ? __ldcg(reinterpret_cast<const float4*>(x0f + e)) : load4_weight<WT>(x0w, e));
      }
    }
    if (ep.epi == EPI_RESID && (rsd0f || rsd0w) && tid < 2 * kMegaPairsMax) sh.rsd[tid] = side;
    if (gsm != nullptr && !mbar_wait(&sh.gbar[gb], static_cast<uint32_t>(guse) & 1u)) {
      atomicOr(a.guard, GUARD_TIMEOUT);
      bad = true;
    }
    if (d.gain != nullptr) {
      // per-group sums of squares (groups <= 4, K <= 4096: the first 4
      // float4 groups of a thread hold its part of x)
      float ssq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = tid * 4 + i * MT * 4;
        if (e < K) {
          const float4 v = xq[i];
          const float t = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
          const int grp = (e >= gsz) + (e >= 2 * gsz) + (e >= 3 * gsz);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (q == grp) ssq[q] += t;
        }
      }
      if (a.groups <= 2) {  // the model's two groups: half the shuffles
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int q = 0; q < 2; ++q) ssq[q] += __shfl_xor_sync(0xffffffffu, ssq[q], o);
      } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int q = 0; q < 4; ++q) ssq[q] += __shfl_xor_sync(0xffffffffu, ssq[q], o);
      }
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
      for (int i = 0; i < 4; ++i) {
        const int e = tid * 4 + i * MT * 4;
        if (e < K) {
          float4 v = xq[i];
          const float rs = sh.rs[(e >= gsz) + (e >= 2 * gsz) + (e >= 3 * gsz)];
          const float4 gn = load4_shared<WT>(gsm, e);
          v.x = v.x * rs * gn.x; v.y = v.y * rs * gn.y; v.z = v.z * rs * gn.z; v.w = v.w * rs * gn.w;
          xq[i] = v;
        }
      }
    }
    if (tiles) {
      // the B fragments of the tile MMAs: per 16 inputs, word (4 h + t) * 2 + r
      // of lane 4 h + t holds inputs 2t + 8r, 2t + 8r + 1 as fp16 (h = 0: high
      // halves, h = 1: low halves)
      uint32_t* xf = reinterpret_cast<uint32_t*>(xs);
#pragma unroll
      for (int i = 0; i < PX; ++i) {
        const int e = tid * 4 + i * MT * 4;
        if (e < KP) {
          const float4 v = xq[i];
          const __half2 h01 = __floats2half2_rn(v.x, v.y), h23 = __floats2half2_rn(v.z, v.w);
          const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
          const __half2 l01 = __floats2half2_rn(v.x - f01.x, v.y - f01.y);
          const __half2 l23 = __floats2half2_rn(v.z - f23.x, v.w - f23.y);
          const int kk = e & 15, t = (kk & 7) >> 1, rr = kk >> 3;
          uint32_t* base = xf + (e >> 4) * 16 + rr;
          base[2 * t] = *reinterpret_cast<const uint32_t*>(&h01);
          base[2 * (t + 1)] = *reinterpret_cast<const uint32_t*>(&h23);
          base[2 * (4 + t)] = *reinterpret_cast<const uint32_t*>(&l01);
          base[2 * (5 + t)] = *reinterpret_cast<const uint32_t*>(&l23);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < PX; ++i) {
        const int e = tid * 4 + i * MT * 4;
        if (e < KP) *reinterpret_cast<float4*>(xs + xidx(e)) = xq[i];
      }
    }
    if (__syncthreads_or(bad)) return false;
  trace_mark(a, q, 1);
  }

  auto finish = [&](int g, float v0, float v1) {
    const int row = 2 * g;
    if (ep.epi == EPI_SWIGLU) {
      st_tagged(ep.out + g, v0 / (1.0f + expf(-v0)) * v1, ep.tag);
    } else if (ep.epi == EPI_QKV) {
      const int half = ep.head_dim / 2;
      const int head = g / half, i = g - head * half;
      float o0 = v0, o1 = v1;
      if (head < ep.n_rot) {
        const float2 cs = sh.rope_pos[i];
        o0 = v0 * cs.x - v1 * cs.y;
        o1 = v1 * cs.x + v0 * cs.y;
      }
      st_tagged(ep.out + head * ep.head_dim + i, o0, ep.tag);
      st_tagged(ep.out + head * ep.head_dim + i + half, o1, ep.tag);
    } else {
      const int rows = min(2, d.N - row);
      const float v[2] = {v0, v1};
      for (int rr = 0; rr < rows; ++rr) {
        if (ep.epi == EPI_RESID) {
          const float nv = sh.rsd[row + rr - 2 * P0] + v[rr];
          sh.rsd[row + rr - 2 * P0] = nv;
          st_tagged(ep.out + row + rr, nv, ep.tag);
          if (ep.plain) ep.plain[row + rr] = nv;
        } else {
          if (ep.logits) ep.logits[row + rr] = v[rr];
          if (v[rr] != v[rr]) atomicOr(ep.guard, GUARD_NAN);
          else best = better(best, Best{v[rr], row + rr});
        }
      }
    }
  };

  if (tiles) {
    // tiles: unit (tile gi of the CTA's range, block b); lane 4 g + t
    // accumulates rows g and g + 8 of the tile -- pair 8 gi + g -- in acc0 / acc1
    // (meaningful for t = 0; fp8: scaled by the rows' scales when the tile
    // ends); a tile split between warps leaves records of its 8 pairs, summed
    // in warp order below
    const uint32_t* xf = reinterpret_cast<const uint32_t*>(xs);
    constexpr int TP = kQ4GroupRows / 2;  // pairs per tile
    const int g8 = lane >> 2;
    float(*recv)[2][TP][2] = reinterpret_cast<float(*)[2][TP][2]>(sh.qs);
    int gi = r.ua / CT, b = r.ua - (r.ua / CT) * CT;
    bool whole = (b == 0);
    float acc0 = 0.f, acc1 = 0.f;
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
#pragma unroll 2
      for (int j = 0; j < n; ++j) {
        const uint8_t* ub = buf + j * UNIT;
        const uint32_t* xb = xf + b * 64;  // the block's four 16-input B fragments
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};  // two MMA chains
        if constexpr (Q4) {
          const uint4 cw = *reinterpret_cast<const uint4*>(ub + lane * 16);
          const float2 sc = *reinterpret_cast<const float2*>(ub + 512 + g8 * 8);
          q4_tile_mma(cw.x, xb, lane, d0);
          q4_tile_mma(cw.y, xb + 16, lane, d1);
          q4_tile_mma(cw.z, xb + 32, lane, d0);
          q4_tile_mma(cw.w, xb + 48, lane, d1);
          acc0 = fmaf(sc.x, (d0[0] + d0[1]) + (d1[0] + d1[1]), acc0);
          acc1 = fmaf(sc.y, (d0[2] + d0[3]) + (d1[2] + d1[3]), acc1);
        } else {
          const uint4 c01 = *reinterpret_cast<const uint4*>(ub + lane * 16);
          const uint4 c23 = *reinterpret_cast<const uint4*>(ub + 512 + lane * 16);
          f8_tile_mma(c01.x, c01.y, xb, lane, d0);
          f8_tile_mma(c01.z, c01.w, xb + 16, lane, d1);
          f8_tile_mma(c23.x, c23.y, xb + 32, lane, d0);
          f8_tile_mma(c23.z, c23.w, xb + 48, lane, d1);
          acc0 += (d0[0] + d0[1]) + (d1[0] + d1[1]);
          acc1 += (d0[2] + d0[3]) + (d1[2] + d1[3]);
        }
        ++b;
        const bool tile_end = (b == CT);
        if (tile_end || u0 + j + 1 == r.ub) {
          const int pl = gi * TP + g8;  // the pair within the CTA's pairs
          if (d.scale != nullptr && (lane & 3) == 0 && P0 + pl < npairs) {  // fp8 row scales
            acc0 *= __ldg(d.scale + 2 * (P0 + pl));
            acc1 *= __ldg(d.scale + 2 * (P0 + pl) + 1);
          }
          if (whole && tile_end) {
            if ((lane & 3) == 0 && P0 + pl < npairs) finish(P0 + pl, acc0, acc1);
          } else {
            const int rr = sh.rec_n[warp];
            if ((lane & 3) == 0) {
              recv[warp][rr][g8][0] = acc0;
              recv[warp][rr][g8][1] = acc1;
            }
            __syncwarp();
            if (lane == 0) {
              sh.rec_pair[warp][rr] = gi;
              sh.rec_n[warp] = rr + 1;
            }
            __syncwarp();
          }
          acc0 = acc1 = 0.f;
          if (tile_end) {
            ++gi;
            b = 0;
            whole = true;
          }
        }
      }
      __syncwarp();  // the slot was only read: no proxy fence needed before refilling it
      ++consumed;
      if (lane == 0) st.issue_next(a, ring, sh.full[warp], cta, G, warp, pos, qkv_n);
    }
    if (bad && lane == 0) atomicOr(a.guard, GUARD_TIMEOUT);
    __syncthreads();
    trace_mark(a, q, 2);
    // split tiles: thread (w, rr, p) of the first record of a tile sums that
    // tile's records of pair p in warp order and finishes the pair
    if (tid < MW * 2 * TP) {
      const int w = tid / (2 * TP), rr = (tid / TP) & 1, p = tid % TP;
      if (rr < sh.rec_n[w]) {
        const int gid = sh.rec_pair[w][rr];
        bool first = true;
        for (int w2 = 0; w2 <= w; ++w2)
          for (int r2 = 0; r2 < sh.rec_n[w2]; ++r2)
            if ((w2 < w || r2 < rr) && sh.rec_pair[w2][r2] == gid) first = false;
        if (first) {
          float v0 = 0.f, v1 = 0.f;
          for (int w2 = w; w2 < MW; ++w2)
            for (int r2 = (w2 == w ? rr : 0); r2 < sh.rec_n[w2]; ++r2)
              if (sh.rec_pair[w2][r2] == gid) {
                v0 += recv[w2][r2][p][0];
                v1 += recv[w2][r2][p][1];
              }
          const int pl = gid * TP + p;
          if (P0 + pl < npairs) finish(P0 + pl, v0, v1);
        }
      }
    }
  } else {
    int pl = r.ua / CT, c = r.ua - (r.ua / CT) * CT;
    bool pair_whole = (c == 0);
    float acc0 = 0.f, acc1 = 0.f;
    // fp8: the current pair's row scales, loaded when the pair starts (used at its end)
    float sc0 = 1.f, sc1 = 1.f;
    if (d.scale && r.ub > r.ua) {
      sc0 = __ldg(d.scale + 2 * (r.p0 + pl));
      sc1 = __ldg(d.scale + 2 * (r.p0 + pl) + 1);
    }
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
          const uint8_t* ub = buf + (j + q) * UNIT;
          if constexpr (Q4) {
            // int4 pair units: the lane's 16 weights are a quarter of one
            // 64-weight block of each row: two partial sums per row, then the
            // block scales
            static_assert(EPL == 16 && UNIT == 576, "int4 unit: 256 code bytes and 8 scales per row");
            const uint2 c0 = *reinterpret_cast<const uint2*>(ub + lane * 8);
            const uint2 c1 = *reinterpret_cast<const uint2*>(ub + 256 + lane * 8);
            const float bs0 = *reinterpret_cast<const float*>(ub + 512 + (lane >> 2) * 4);
            const float bs1 = *reinterpret_cast<const float*>(ub + 544 + (lane >> 2) * 4);
            f32x2 p00 = 0ull, p01 = 0ull, p10 = 0ull, p11 = 0ull;  // (row, word) sums of element pairs
            q4_dot8(c0.x, xv, p00);
            q4_dot8(c0.y, xv + 8, p01);
            q4_dot8(c1.x, xv, p10);
            q4_dot8(c1.y, xv + 8, p11);
            acc0 = fmaf(sum2(p00) + sum2(p01), bs0, acc0);
            acc1 = fmaf(sum2(p10) + sum2(p11), bs1, acc1);
          } else {
            const uint8_t* u8 = ub + lane * 16;
            float w0[EPL], w1[EPL];
            Unpack<PT>::run(*reinterpret_cast<const uint4*>(u8), w0);
            Unpack<PT>::run(*reinterpret_cast<const uint4*>(u8 + 512), w1);
            f32x2 t0 = 0ull, t1 = 0ull;  // sums of element pairs
#pragma unroll
            for (int e = 0; e < EPL; e += 2) {
              const f32x2 xe = pk2(xv[e], xv[e + 1]);
              t0 = fma2(pk2(w0[e], w0[e + 1]), xe, t0);
              t1 = fma2(pk2(w1[e], w1[e + 1]), xe, t1);
            }
            acc0 += sum2(t0);
            acc1 += sum2(t1);
          }
        }
        j += seg;
        c += seg;
        const bool pair_end = (c == CT);
        const bool range_end = (u0 + j == r.ub);
        if (pair_end || range_end) {
          const float s0 = warp_sum(acc0) * sc0, s1 = warp_sum(acc1) * sc1;
          acc0 = acc1 = 0.f;
          if (lane == 0) {
            if (pair_whole && pair_end) {
              finish(P0 + pl, s0, s1);
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
            if (d.scale && r.ua + (u0 - r.ua) + j < r.ub) {
              sc0 = __ldg(d.scale + 2 * (r.p0 + pl));
              sc1 = __ldg(d.scale + 2 * (r.p0 + pl) + 1);
            }
          }
        }
      }
      __syncwarp();  // the slot was only read: no proxy fence needed before refilling it
      ++consumed;
      if (lane == 0) st.issue_next(a, ring, sh.full[warp], cta, G, warp, pos, qkv_n);
    }
    if (bad && lane == 0) atomicOr(a.guard, GUARD_TIMEOUT);
    __syncthreads();
    trace_mark(a, q, 2);
    // Pairs split between warps: at most two records per warp, lane 2w + rr of
    // warp 0 holding record rr of warp w.  Every record of a pair is summed in
    // warp order by the lane of its first record, which finishes the pair; a
    // fixed 16-step shuffle loop, so the lanes never diverge.
    if (warp == 0) {
      const int w = lane >> 1, rr = lane & 1;
      const bool has = lane < 2 * MW && rr < sh.rec_n[w];
      const int pr = has ? sh.rec_pair[w][rr] : -1 - lane;
      const float a0 = has ? sh.rec_val[w][rr][0] : 0.f, a1 = has ? sh.rec_val[w][rr][1] : 0.f;
      float v0 = 0.f, v1 = 0.f;
      bool first = has;
#pragma unroll
      for (int j = 0; j < 2 * MW; ++j) {
        const int pj = __shfl_sync(0xffffffffu, pr, j);
        const float b0 = __shfl_sync(0xffffffffu, a0, j), b1 = __shfl_sync(0xffffffffu, a1, j);
        if (pj == pr) {
          if (j < lane) first = false;
          if (j >= lane) {
            v0 += b0;
            v1 += b1;
          }
        }
      }
      if (first) finish(P0 + pr, v0, v1);
    }
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

// One attention item (KV head g, key split sp) per CTA: the partial
// (max, sum, unnormalised output) of its REP query heads over its keys; the
// last split of head g to finish merges all splits into attn_out.
template <typename WT, int D, int REP, int UB, typename KVT>
__device__ bool a_phase(const MegaArgs& a, int l, int pos, uint32_t tag_in, uint32_t tag_out, uint8_t* smem,
                        MegaShared& sh, Stream<UB, D, KVT>& st, int& consumed, int cta, int G, int qkv_n) {
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
  constexpr int NQ4 = ((REP + 2) * D + MT - 1) / MT;  // tagged words per thread to stage
  static_assert(TKM > 0 && 2 * KVB + 2 * TKM * 2 <= SB, "an attention tile must fit one slot");
  static_assert(D <= 128 && REP * D <= 512, "staging buffers");
  static_assert(REP <= MW, "one warp per query head in the merge");
  constexpr bool TCA = tc_attn<D, KVT>();
  __shared__ float wstate[MW][PSTR];
  __shared__ float wfac[MW][REP];  // per warp and query head: exp(m_warp - m_split)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (cta >= a.nkv * a.nsplit) return true;
  const int L = pos + 1;
  const AItem it = a_item<TKM>(sh);
  const int nmine = a_mine<TKM>(it, warp);
  const size_t head_row = (static_cast<size_t>(a.seq) * a.nkv + it.g) * a.cap;
  uint8_t* ring = smem + static_cast<size_t>(warp) * NS * SB;
  const bool appends = (it.k1 == L);  // this split holds the new token's key

  // ---- stage the query heads (and the new K/V rows) once their tags arrive
  {
    const int total = REP * D + (appends ? 2 * D : 0);
    const u64* src[NQ4];
    unsigned pend = 0;
#pragma unroll
    for (int i = 0; i < NQ4; ++i) {
      const int idx = tid + i * MT;
      src[i] = a.t_qkv;
      if (idx < total) {
        pend |= 1u << i;
        if (idx < REP * D) {
          src[i] = a.t_qkv + static_cast<size_t>(it.g) * REP * D + idx;
        } else {
          const int kv = (idx - REP * D) / D, e = (idx - REP * D) - kv * D;
          src[i] = a.t_qkv + (kv == 0 ? a.nq * D : (a.nq + a.nkv) * D) + it.g * D + e;
        }
      }
    }
    Patience wait(a.poll_limit_ns);
    bool bad = false;
    while (pend) {
      u64 w[NQ4];
#pragma unroll
      for (int i = 0; i < NQ4; ++i) w[i] = (pend & (1u << i)) ? ld_tagged(src[i]) : 0ull;
#pragma unroll
      for (int i = 0; i < NQ4; ++i) {
        if ((pend & (1u << i)) && tag_is(w[i], tag_in)) {
          const int idx = tid + i * MT;
          if (idx < REP * D) sh.qs[idx] = tag_val(w[i]) * a.scale;
          else sh.newkv[(idx - REP * D) / D][(idx - REP * D) % D] = tag_val(w[i]);
          pend &= ~(1u << i);
        }
      }
      if (pend && !wait.more(a.guard)) {
        bad = true;
        break;
      }
    }
    if (__syncthreads_or(bad)) return false;
  }
  trace_mark(a, l * kPhases + PH_ATTN, 1);
  bool bad = false;
  if constexpr (!TCA) {
  __shared__ float Sw[MW][REP][TKM];
  __shared__ __align__(16) float Pw[MW][TKM][REP];
  const int kl = lane % LPK;
  float q[REP][QD];
#pragma unroll
  for (int h = 0; h < REP; ++h)
#pragma unroll
    for (int e = 0; e < QD; ++e) q[h][e] = sh.qs[h * D + kl * QD + e];

  float m[REP], lsum[REP], acc[REP][DPL];
#pragma unroll
  for (int h = 0; h < REP; ++h) {
    m[h] = -INFINITY;
    lsum[h] = 0.f;
#pragma unroll
    for (int dd = 0; dd < DPL; ++dd) acc[h][dd] = 0.f;
  }
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
    if (appends && jr >= 0 && jr < rows) {  // the new token: cache format, to global and into the slot
      for (int kv = 0; kv < 2; ++kv) {
        const float* src = sh.newkv[kv];
        KVT* dst = reinterpret_cast<KVT*>((kv == 0 ? a.kc : a.vc) + static_cast<size_t>(l) * a.s_kv) +
                   (head_row + pos) * D;
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
            reinterpret_cast<__half*>((kv == 0 ? a.ks : a.vs) + static_cast<size_t>(l) * a.s_sc)[head_row + pos] = sh16;
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
    // scores: 8 lanes per key, every step computed (rows past the end hold
    // stale bytes of the slot; their scores are never stored), so the
    // compiler can overlap the steps
#pragma unroll
    for (int stp = 0; stp < (TKM + KPS - 1) / KPS; ++stp) {
      const int jj = stp * KPS + lane / LPK;
      float dot[REP];
#pragma unroll
      for (int h = 0; h < REP; ++h) dot[h] = 0.f;
      {
        const uint8_t* kr = slot + min(jj, TKM - 1) * ROWB + kl * VPL * 16;
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
    // online softmax over the tile, lane = key, the REP heads interleaved
    float al[REP], pr[REP], ps[REP];
#pragma unroll
    for (int h = 0; h < REP; ++h) {
      const float sv = lane < rows ? Sw[warp][h][lane] : -INFINITY;
      const float mn = fmaxf(m[h], warp_max_redux(sv));
      al[h] = expf(m[h] - mn);
      pr[h] = lane < rows ? expf(sv - mn) : 0.f;
      ps[h] = pr[h];
      m[h] = mn;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int h = 0; h < REP; ++h) ps[h] += __shfl_xor_sync(0xffffffffu, ps[h], o);
    const float vs_l = I8 && lane < rows ? __half2float(vsc[lane]) : 1.f;
#pragma unroll
    for (int h = 0; h < REP; ++h) {
      lsum[h] = lsum[h] * al[h] + ps[h];
      if (lane < rows) Pw[warp][lane][h] = pr[h] * vs_l;
    }
    __syncwarp();
    if (lane < DL) {
#pragma unroll
      for (int h = 0; h < REP; ++h)
#pragma unroll
        for (int dd = 0; dd < DPL; ++dd) acc[h][dd] *= al[h];
      const KVT* vt = reinterpret_cast<const KVT*>(slot + KVB) + lane * DPL;
      auto pv_row = [&](int jj) {
        float vf[DPL];
        vload<DPL>(vt + jj * D, vf);
        float pw[REP];
        if constexpr (REP == 4) {
          const float4 p4 = *reinterpret_cast<const float4*>(&Pw[warp][jj][0]);
          pw[0] = p4.x; pw[1] = p4.y; pw[2] = p4.z; pw[3] = p4.w;
        } else {
#pragma unroll
          for (int h = 0; h < REP; ++h) pw[h] = Pw[warp][jj][h];
        }
#pragma unroll
        for (int h = 0; h < REP; ++h)
#pragma unroll
          for (int dd = 0; dd < DPL; ++dd) acc[h][dd] = fmaf(pw[h], vf[dd], acc[h][dd]);
      };
      if (rows == TKM) {  // a full tile: every row, unrolled
#pragma unroll
        for (int jj = 0; jj < TKM; ++jj) pv_row(jj);
      } else {
        for (int jj = 0; jj < rows; ++jj) pv_row(jj);
      }
    }
    // Where this slot was written by generic stores (the new row), order
    // those writes before the next bulk copy into it.  Slots that were only
    // read need no proxy fence: every load has completed (its value was used)
    // before the warp barrier, as with a consumer-release mbarrier.
    if (appends && jr >= 0 && jr < rows) fence_proxy_async();
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
  } else {
  // Q.K^T and P.V on the tensor cores (mma.sync m16n8k16, fp16 operands,
  // fp32 accumulation).  M rows: row h < REP is fp16(q_h) (or fp16(p_h)), row
  // REP + h the remainder q_h - fp16(q_h), so one MMA carries both halves; the
  // fp16 K/V values are exact.  The tile's boxes are swizzled (chunk c of row r
  // at c ^ (r & 7)), so the ldmatrix loads hit distinct banks.
  constexpr int NB = D / 64, KS = D / 16, NT = D / 8, XR = 4 * REP;
  static_assert(TKM == 16 && (REP == 1 || REP == 2 || REP == 4), "tensor-core tile shape");
  const int gq = lane >> 2, tq = lane & 3, hq = gq % REP;
  const bool live = gq < 2 * REP, rem = gq >= REP;
  uint32_t qa[KS][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int d = 16 * ks + 8 * hf + 2 * tq;
      uint32_t hi = 0u, lo = 0u;
      if (live) split_half2(sh.qs[hq * D + d], sh.qs[hq * D + d + 1], hi, lo);
      qa[ks][hf] = rem ? lo : hi;
    }
  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
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
    uint8_t* ksl = ring + static_cast<size_t>(s) * SB;
    uint8_t* vsl = ksl + NB * kTcBox;
    const int jr = pos - j0;
    const bool newrow = appends && jr >= 0 && jr < rows;
    if (newrow) {  // the new token: fp16 to the cache and into the swizzled slot
      for (int kv = 0; kv < 2; ++kv) {
        const float* src = sh.newkv[kv];
        __half* dst = reinterpret_cast<__half*>((kv == 0 ? a.kc : a.vc) + static_cast<size_t>(l) * a.s_kv) +
                      (head_row + pos) * D;
        uint8_t* base = kv == 0 ? ksl : vsl;
        for (int e = lane; e < D; e += 32) {
          const __half hv = __float2half_rn(src[e]);
          dst[e] = hv;
          *reinterpret_cast<__half*>(base + (e >> 6) * kTcBox + swz128(jr, (e & 63) >> 3) + (e & 7) * 2) = hv;
        }
      }
    }
    if (rows < TKM) {  // stale rows past the tile: P is 0 there, but 0 x NaN is NaN
      for (int e = lane; e < (TKM - rows) * NB * 8; e += 32) {
        const int r = rows + e / (NB * 8), bx = (e / 8) % NB, c = e & 7;
        *reinterpret_cast<uint4*>(vsl + bx * kTcBox + r * 128 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    __syncwarp();
    float sacc[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint32_t af[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
      const int mi = lane >> 3, key = 8 * (mi >> 1) + (lane & 7), chunk = 2 * ks + (mi & 1);
      uint32_t r0, r1, r2, r3;
      ldsm_x4(smem_u32(ksl + (chunk >> 3) * kTcBox + swz128(key, chunk & 7)), r0, r1, r2, r3);
      mma16816(sacc[0], af, r0, r1);
      mma16816(sacc[1], af, r2, r3);
    }
    // this lane's row: keys 8n + 2tq + e; the two halves of q add up
    float sc[2][2];
    float mx = -INFINITY;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float v = sacc[n][e] + __shfl_xor_sync(0xffffffffu, sacc[n][e], XR);
        sc[n][e] = 8 * n + 2 * tq + e < rows ? v : -INFINITY;
        mx = fmaxf(mx, sc[n][e]);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m_run, mx);
    const float al = expf(m_run - mn);
    float ps = 0.f;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[n][e] = expf(sc[n][e] - mn);
        ps += sc[n][e];
      }
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    l_run = l_run * al + ps;
    m_run = mn;
    uint32_t pa[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t hi = 0u, lo = 0u;
      if (live) split_half2(sc[hf][0], sc[hf][1], hi, lo);
      pa[hf] = rem ? lo : hi;
    }
    const uint32_t pf[4] = {pa[0], 0u, pa[1], 0u};
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      const int mi = lane >> 3, key = 8 * (mi & 1) + (lane & 7), chunk = 2 * np + (mi >> 1);
      uint32_t r0, r1, r2, r3;
      ldsm_x4_t(smem_u32(vsl + (chunk >> 3) * kTcBox + swz128(key, chunk & 7)), r0, r1, r2, r3);
      o[2 * np][0] *= al;
      o[2 * np][1] *= al;
      o[2 * np + 1][0] *= al;
      o[2 * np + 1][1] *= al;
      mma16816(o[2 * np], pf, r0, r1);
      mma16816(o[2 * np + 1], pf, r2, r3);
    }
    // generic stores into the slot (the new row, zeroed rows) before the next copy over them
    if (newrow || rows < TKM) fence_proxy_async();
    __syncwarp();
    ++consumed;
    if (lane == 0) st.issue_next(a, ring, sh.full[warp], cta, G, warp, pos, qkv_n);
  }
  if (bad && lane == 0) atomicOr(a.guard, GUARD_TIMEOUT);
  if (live && !rem && tq == 0) {
    wstate[warp][hq] = m_run;
    wstate[warp][REP + hq] = l_run;
  }
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float v = o[n][e] + __shfl_xor_sync(0xffffffffu, o[n][e], XR);
      if (live && !rem) wstate[warp][2 * REP + hq * D + 8 * n + 2 * tq + e] = v;
    }
  }
  if (__syncthreads_or(bad)) return false;
  trace_mark(a, l * kPhases + PH_ATTN, 2);
  // ---- this split's partial (max, sum, unnormalised output per query head):
  // combine the warps and publish it as tagged words.  Then every split of
  // the KV head merges one slice of the REP * D outputs from all the splits'
  // partials, so each CTA reads a few hundred words instead of one CTA
  // reading them all.
  const int ns = a.nsplit;
  float* stage = reinterpret_cast<float*>(smem + kMegaRingBytes);  // the x buffer is free here
  u64* pub = a.t_part + static_cast<size_t>(cta) * PSTR;
  if (tid < MW * REP) {
    const int w = tid / REP, h = tid - (tid / REP) * REP;
    float M = -INFINITY;
    for (int v = 0; v < MW; ++v) M = fmaxf(M, wstate[v][h]);
    wfac[w][h] = wstate[w][h] == -INFINITY ? 0.f : expf(wstate[w][h] - M);
  }
  __syncthreads();
  for (int idx = tid; idx < REP * D; idx += MT) {
    const int h = idx / D;
    float O = 0.f;
    for (int w = 0; w < MW; ++w) O = fmaf(wstate[w][2 * REP + idx], wfac[w][h], O);
    st_tagged(pub + 2 * REP + idx, O, tag_out);
  }
  if (tid < REP) {
    float M = -INFINITY;
    for (int w = 0; w < MW; ++w) M = fmaxf(M, wstate[w][tid]);
    float Ls = 0.f;
    for (int w = 0; w < MW; ++w) Ls = fmaf(wstate[w][REP + tid], wfac[w][tid], Ls);
    st_tagged(pub + tid, M, tag_out);
    st_tagged(pub + REP + tid, Ls, tag_out);
  }
  // ---- this split's slice [o0, o1) of the merged outputs
  const int o0 = (REP * D * it.sp) / ns, o1 = (REP * D * (it.sp + 1)) / ns, nsl = o1 - o0;
  const u64* head_part = a.t_part + static_cast<size_t>(it.g) * ns * PSTR;  // split s at s * PSTR
  float* mlv = stage;               // [s][2 * REP]: max, then sum, per query head
  float* ov = stage + 2 * REP * ns;  // [s][nsl]: the slice of each split's output
  {
    constexpr int NPW = (2 * REP * kMegaSplitMax + REP * D + kMegaSplitMax + MT - 1) / MT;
    const int nml = 2 * REP * ns, nw = nml + nsl * ns;
    const u64* src[NPW];
    unsigned pend = 0;
#pragma unroll
    for (int i = 0; i < NPW; ++i) {
      const int k = tid + i * MT;
      src[i] = head_part;
      if (k < nw) {
        pend |= 1u << i;
        if (k < nml) {
          const int sp = k / (2 * REP);
          src[i] = head_part + static_cast<size_t>(sp) * PSTR + (k - sp * 2 * REP);
        } else {
          const int kk = k - nml, sp = kk / nsl;
          src[i] = head_part + static_cast<size_t>(sp) * PSTR + 2 * REP + o0 + (kk - sp * nsl);
        }
      }
    }
    Patience wait(a.poll_limit_ns);
    bool bad = false;
    while (pend) {
      u64 w[NPW];
#pragma unroll
      for (int i = 0; i < NPW; ++i) w[i] = (pend & (1u << i)) ? ld_tagged(src[i]) : 0ull;
#pragma unroll
      for (int i = 0; i < NPW; ++i) {
        if ((pend & (1u << i)) && tag_is(w[i], tag_out)) {
          stage[tid + i * MT] = tag_val(w[i]);  // mlv then ov: the word order above
          pend &= ~(1u << i);
        }
      }
      if (pend && !wait.more(a.guard)) {
        bad = true;
        break;
      }
    }
    if (__syncthreads_or(bad)) return false;
  }
  float* wts = &wstate[0][0];  // MW * PSTR >= nsplit * REP floats
  if (warp < REP) {  // warp h, lane per split: the weight of each split, exp(M_s - M) / sum
    const int h = warp;
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, mlv[s * 2 * REP + h]);
    M = warp_max(M);
    float Ls = 0.f;
    for (int s = lane; s < ns; s += 32) {
      const float ms = mlv[s * 2 * REP + h];
      if (ms != -INFINITY) Ls = fmaf(mlv[s * 2 * REP + REP + h], expf(ms - M), Ls);
    }
    Ls = warp_sum(Ls);
    for (int s = lane; s < ns; s += 32) {
      const float ms = mlv[s * 2 * REP + h];
      wts[s * REP + h] = ms == -INFINITY ? 0.f : expf(ms - M) / Ls;
    }
  }
  __syncthreads();
  for (int t = tid; t < nsl; t += MT) {
    const int idx = o0 + t, h = idx / D;
    float O = 0.f;
    for (int s = 0; s < ns; ++s) O = fmaf(ov[s * nsl + t], wts[s * REP + h], O);
    st_tagged(a.t_attn + static_cast<size_t>(it.g) * REP * D + idx, O, tag_out);
  }
  __syncthreads();  // the stage is the next phase's x buffer
  return true;
}

// ---- the step -------------------------------------------------------------------------------
template <typename WT, typename PT, int D, int REP, typename KVT>
__global__ void __launch_bounds__(MT, 1) mega_decode_kernel(const __grid_constant__ KvMaps maps, const MegaArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the tensor-core attention's swizzled boxes need 1024-byte aligned slots
  uint8_t* const smem = tc_attn<D, KVT>() ? reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                                        ~static_cast<uintptr_t>(1023))
                                          : smem_raw;
  __shared__ MegaShared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  const int pos = a.seq_len[a.seq];
  if (pos < 0 || pos >= a.cap) {
    if (tid == 0) atomicOr(a.guard, GUARD_POS);
    return;  // every CTA sees the same pos and leaves before any wait
  }
  const uint32_t tagbase = (*a.epoch + 1u) << kMegaTagShift;
  const int qkv_n = (a.nq + 2 * a.nkv) * D;
  Stream<Fmt<PT>::UNIT, D, KVT> st;
  GainQ gq;
  if (tid == 0) {
    mbar_init(&sh.gbar[0], 1);
    mbar_init(&sh.gbar[1], 1);
  }
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&sh.full[warp][s], 1);
    fence_mbar_init();
  }
  // per-launch tables: row splits of the five GEMV kinds, the attention item,
  // the norm-gain pointers
  if (tid < 5 * MW) {
    const int kind = tid / MW, w = tid - (tid / MW) * MW;
    const int N = kind == 0 ? qkv_n : kind == 2 ? 2 * a.inter : kind == 4 ? a.vocab : a.hidden;
    const int CT = kind == 0 ? a.g_qkv.CT : kind == 1 ? a.g_o.CT : kind == 2 ? a.g_gu.CT
                 : kind == 3 ? a.g_down.CT : a.g_lm.CT;
    // fp8 / int4 tiled kinds own rows in tiles of 16: the split counts tiles as its "pairs"
    const bool tl = (std::is_same<PT, q4_block64>::value || std::is_same<PT, __nv_fp8_e4m3>::value) && tiled_kind(kind);
    sh.wr[kind][w] = g_split(tl ? 2 * ((N + kQ4GroupRows - 1) / kQ4GroupRows) : N, CT, cta, G, w);
  }
  if (tid == 5 * MW) sh.item = a_split(a, min(cta, a.nkv * a.nsplit - 1), pos + 1);
  for (int i = tid; i < 2 * a.n_layers; i += MT)
    sh.gains[i] = (i & 1) ? a.layers[i >> 1].mlp_norm : a.layers[i >> 1].attn_norm;
  __syncthreads();  // barriers initialised, tables written
  if (lane == 0)
    st.start(a, sh, &maps, smem + static_cast<size_t>(warp) * NS * SB, sh.full[warp], cta, G, warp, pos, qkv_n);
  if (tid == 0) issue_gain(a, smem, sh, gq, sh.gains[0], a.hidden * static_cast<int>(sizeof(WT)));
  if (tid < D / 2) sh.rope_pos[tid] = a.rope[static_cast<size_t>(pos) * (D / 2) + tid];
  int consumed = 0;
  Best best{-INFINITY, 0x7fffffff};
  if (a.trace != nullptr && tid == 0) {  // aligns this SM's clock with the others
    const size_t at = (static_cast<size_t>(a.n_layers * kPhases + 1) * G + cta) * 4;
    a.trace[at] = globaltimer();
    a.trace[at + 1] = sm_clock();
  }

  const WT* xe = nullptr;
  if (!a.x_ext) {
    const int tok = *a.token_in;
    if (a.hist && cta == 0 && tid == 0) a.hist[static_cast<size_t>(a.seq) * a.cap + pos] = tok;
    if (tok < 0 || tok >= a.vocab) {
      if (tid == 0) atomicOr(a.guard, GUARD_TOKEN);
      xe = static_cast<const WT*>(a.embed);  // row 0 stands in; the guard reports the fault
    } else {
      xe = static_cast<const WT*>(a.embed) + static_cast<size_t>(tok) * a.hidden;
    }
  }

  // One loop over the phases, so that each phase body exists once in the
  // code: the instruction cache stays warm from one phase to the next.
  // Phase q reads what phase q - 1 wrote.
  const int lastq = a.n_layers * kPhases - 1 + (a.head ? 1 : 0);
  bool ok = true;
  for (int q = 0; q <= lastq && ok; ++q) {
    const int l = q / kPhases, j = q - (q / kPhases) * kPhases;
    uint32_t tag_in = tagbase | static_cast<uint32_t>(q - 1);
    const uint32_t tag_out = tagbase | static_cast<uint32_t>(q);
    if (q == a.stall_phase) tag_in = tagbase | ((1u << kMegaTagShift) - 1u);  // no phase has this number
    if (lane == 0 && a.l2_ahead > 0 && ((a.l2_mask >> (l < a.n_layers ? j : 5)) & 1))
      stream_prefetch(st, a, cta, G, warp, pos, qkv_n, a.l2_ahead);
    trace_mark(a, q, 0);
    if (l < a.n_layers && j == PH_ATTN) {
      ok = a_phase<WT, D, REP>(a, l, pos, tag_in, tag_out, smem, sh, st, consumed, cta, G, qkv_n);
      trace_mark(a, q, 3);
      continue;
    }
    GEpi ep{EPI_RESID, a.t_resid, nullptr, a.rope, pos, D, a.nq + a.nkv, nullptr, a.guard, tag_out};
    const u64* xt = a.t_resid;
    const float* x0f = nullptr;
    const WT* x0w = nullptr;
    const float* r0f = nullptr;
    const WT* r0w = nullptr;
    if (l >= a.n_layers) {
      ep.epi = EPI_ARGMAX;
      ep.out = nullptr;
      ep.logits = a.logits;
    } else if (j == PH_QKV) {
      ep.epi = EPI_QKV;
      ep.out = a.t_qkv;
      if (l == 0) {
        xt = nullptr;
        x0f = a.x_ext;
        x0w = xe;
      }
    } else if (j == PH_O) {
      xt = a.t_attn;
      if (l == 0) {  // the residual rows start as the layer input
        r0f = a.x_ext;
        r0w = xe;
      }
    } else if (j == PH_GU) {
      ep.epi = EPI_SWIGLU;
      ep.out = a.t_act;
    } else {
      xt = a.t_act;
      if (l == a.n_layers - 1) ep.plain = a.x_out;
    }
    ok = g_phase<WT, PT, D, KVT>(a, q, gdesc(a, sh, q, qkv_n, D), xt, tag_in, x0f, x0w, r0f, r0w, ep, smem, sh, st,
                                 gq, consumed, best, cta, G, pos, qkv_n);
    trace_mark(a, q, 3);
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
  if (tid == 0) {
    for (int k = gq.used; k < gq.issued; ++k)
      if (!mbar_wait(&sh.gbar[k & 1], static_cast<uint32_t>(k >> 1) & 1u)) break;
  }
  // the last CTA to get here finishes the step and re-arms the counters
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
    *a.end_count = 0u;
    *a.epoch = *a.epoch + 1u;  // the next launch writes fresh tags
  }
}

template <int D, typename KVT>
constexpr bool tile_fits() {
  return tile_keys<D, KVT>() > 0;
}

template <typename WT, typename PT, int D, int REP, typename KVT>
const void* mega_fn() {
  if constexpr (tile_fits<D, KVT>())
    return reinterpret_cast<const void*>(mega_decode_kernel<WT, PT, D, REP, KVT>);
  else
    return nullptr;
}

// (gain / embedding type, packed weight type and its format key, head_dim,
// GQA ratio) combinations with a persistent kernel: the 3.7B shape and the
// medium model in bf16, fp8 and int4 weights, the tiny fp32 model
#define K2_MEGA_SHAPES(X)                                                                                         \
  X(__nv_bfloat16, __nv_bfloat16, 2, 128, 4) X(__nv_bfloat16, __nv_bfloat16, 2, 64, 4) X(float, float, 4, 16, 2) \
  X(__nv_bfloat16, __nv_fp8_e4m3, 1, 128, 4) X(__nv_bfloat16, __nv_fp8_e4m3, 1, 64, 4)                           \
  X(__nv_bfloat16, q4_block64, kWfmtQ4, 128, 4) X(__nv_bfloat16, q4_block64, kWfmtQ4, 64, 4)

// wfmt: the packed weight format (kWfmt* in k2_kernels.h)
const void* mega_lookup(int wfmt, int head_dim, int rep, int kv_dtype) {
#define K2_MEGA_LOOK(WT, PT, WB, D, R)                               \
  if (wfmt == WB && head_dim == D && rep == R) {                     \
    if (kv_dtype == 0) return mega_fn<WT, PT, D, R, float>();        \
    if (kv_dtype == 2) return mega_fn<WT, PT, D, R, __half>();       \
    if (kv_dtype == 3) return mega_fn<WT, PT, D, R, int8_t>();       \
  }
  K2_MEGA_SHAPES(K2_MEGA_LOOK)
#undef K2_MEGA_LOOK
  return nullptr;
}

}  // namespace

bool mega_supported(int wfmt, int head_dim, int rep, int kv_dtype) {
  return mega_lookup(wfmt, head_dim, rep, kv_dtype) != nullptr;
}

bool mega_tc_attention(int head_dim, int kv_dtype) { return kv_dtype == 2 && head_dim % 64 == 0; }

namespace {
// dynamic shared memory of an instance: the tensor-core attention aligns its ring to 1024 bytes
size_t mega_smem(int head_dim, int kv_dtype) { return kMegaSmemBytes + (mega_tc_attention(head_dim, kv_dtype) ? 1024 : 0); }
}  // namespace

cudaError_t mega_init_attrs(int wfmt, int head_dim, int rep, int kv_dtype) {
  const void* fn = mega_lookup(wfmt, head_dim, rep, kv_dtype);
  if (!fn) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(mega_smem(head_dim, kv_dtype)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                              static_cast<int>(cudaSharedmemCarveoutMaxShared));
}

int mega_max_grid(int wfmt, int head_dim, int rep, int kv_dtype) {
  const void* fn = mega_lookup(wfmt, head_dim, rep, kv_dtype);
  if (!fn) return 0;
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, MT, mega_smem(head_dim, kv_dtype)) != cudaSuccess)
    return 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return per_sm >= 1 ? sms : 0;  // one CTA per SM
}

cudaError_t launch_mega(const MegaArgs& a, const KvMaps& maps, int wfmt, int head_dim, int rep, int kv_dtype, int grid,
                        cudaStream_t s) {
  const void* fn = mega_lookup(wfmt, head_dim, rep, kv_dtype);
  if (!fn) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MT);
  cfg.dynamicSmemBytes = mega_smem(head_dim, kv_dtype);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<KvMaps*>(&maps), const_cast<MegaArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace k2
