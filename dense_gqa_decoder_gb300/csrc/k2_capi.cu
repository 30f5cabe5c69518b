// Host side of libk2: config validation, workspace layout, the decode-step
// launch sequence, graph caching, and the C ABI declared in include/k2.h.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>
#include <stddef.h>
#include <cmath>
#include <cstring>

#include <algorithm>
#include <array>
#include <map>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/k2.h"
#include "k2_kernels.h"

using namespace k2;

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kGemvSmem = 104 * 1024;  // per-CTA budget: CTAs of two consecutive kernels share one SM
constexpr size_t kLmHeadSmem = 176 * 1024;
constexpr int kArgmaxPartsMax = 1024;
constexpr int kPrefillChunk = 2048;  // prompt tokens per tensor-core prefill pass
constexpr int kTcPrefillMin = 8;     // shorter prompts are appended one decode step per token
constexpr int kSpecMax = 8;          // drafted ids verified in one pass

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int elt_bytes(int dt) { return dt == K2_F32 ? 4 : (dt == K2_BF16 || dt == K2_F16) ? 2 : 1; }

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
struct Layout {
  size_t seq_len, guard, am_counter, msync, rope, resid, qkv, attn_out, act, am_val, am_idx, attn_part, ltab;
  size_t t_resid, t_qkv, t_attn, t_act, t_part;  // persistent step: (value, tag) activations
  size_t hist, slog, sscr, sample_row;             // token history, sampling logits and scratch
  size_t sqkv, so, sgu, sdown, slm;                // fp8 weights: per-row scales (first layer)
  size_t sqkv_layer, so_layer, sgu_layer, sdown_layer;
  size_t dq[4], dq_bytes[4];  // int4 prefill: matrix m of the current layer, bf16 hi then lo
  size_t w16[2][4];           // bf16 weights, fp16 prefill: matrix m of layers of parity 0 / 1 as fp16
  size_t vlog, vids, varg, vpv, vpi;               // speculative verification: logits, ids, argmax
  // tensor-core prefill of up to `pchunk` tokens at a time (bf16 weights)
  int pchunk;
  size_t px, pxh, pxl, pah, pal, pqkv, pq, plog;
  size_t wqkv, wo, wgu, wdown, wlm;  // packed weights; per-layer strides below
  size_t wqkv_layer, wo_layer, wgu_layer, wdown_layer;
  // fp8 weights with a tensor-core prefill: the codes as bf16 in the bf16 packed layout
  size_t tqkv, to, tgu, tdown;
  size_t tqkv_layer, to_layer, tgu_layer, tdown_layer;
  size_t kc, vc, ks, vs;  // first layer; per-layer stride kv_layer / sc_layer
  size_t kv_layer, sc_layer;
  size_t total;
  size_t repack_bytes, kv_bytes;
  int cap;
};

struct Sizes {
  int H, L, nq, nkv, d, I, G, V, ctx, B, qkv_n, rep, wb, kvb;
  int gb;  // bytes of an embedding / gain element (bf16 for fp8 / int4 weights); wb: of a packed weight
  int wf;  // the packed weight format key of the persistent step (kWfmt*: weight bytes, or kWfmtQ4)
};

bool quantized(int weight_dtype) { return weight_dtype == K2_F8 || weight_dtype == K2_Q4; }

Sizes sizes_of(const k2_config& c) {
  Sizes s;
  s.H = c.hidden; s.L = c.n_layers; s.nq = c.n_heads; s.nkv = c.n_kv_heads; s.d = c.head_dim;
  s.I = c.intermediate; s.G = c.norm_groups; s.V = c.vocab; s.ctx = c.max_context; s.B = c.max_batch;
  s.qkv_n = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  s.rep = c.n_kv_heads > 0 ? c.n_heads / c.n_kv_heads : 0;
  s.wb = elt_bytes(c.weight_dtype);
  s.gb = quantized(c.weight_dtype) ? 2 : s.wb;
  s.wf = c.weight_dtype == K2_Q4 ? kWfmtQ4 : s.wb;
  s.kvb = elt_bytes(c.kv_dtype);
  return s;
}

Layout layout_of(const k2_config& c) {
  const Sizes s = sizes_of(c);
  Layout l = {};
  // rows of KV per sequence: room for max_context rows plus the 16-byte
  // rounding of int8 scale copies, in whole 64-row tiles
  l.cap = static_cast<int>(align_up(static_cast<size_t>(s.ctx) + 8, 64));
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, kAlign);
    return at;
  };
  l.seq_len = take(sizeof(int) * s.B);
  l.guard = take(sizeof(unsigned));
  l.am_counter = take(sizeof(unsigned) * s.B);
  // persistent step: finished CTAs, launch epoch
  l.msync = take(sizeof(unsigned) * 2);
  l.rope = take(sizeof(float2) * static_cast<size_t>(l.cap) * (s.d / 2));
  l.resid = take(sizeof(float) * static_cast<size_t>(s.B) * s.H);
  l.qkv = take(sizeof(float) * static_cast<size_t>(s.B) * s.qkv_n);
  l.attn_out = take(sizeof(float) * static_cast<size_t>(s.B) * s.nq * s.d);
  l.act = take(sizeof(float) * static_cast<size_t>(s.B) * s.I);
  l.am_val = take(sizeof(float) * static_cast<size_t>(s.B) * kArgmaxPartsMax);
  l.am_idx = take(sizeof(int) * static_cast<size_t>(s.B) * kArgmaxPartsMax);
  l.attn_part = take(sizeof(float) * static_cast<size_t>(s.nkv) * kMegaSplitMax * s.rep * (s.d + 2));
  l.ltab = take(sizeof(LayerPtrs) * static_cast<size_t>(s.L));
  l.t_resid = take(8 * static_cast<size_t>(s.H));
  l.t_qkv = take(8 * static_cast<size_t>(s.qkv_n));
  l.t_attn = take(8 * static_cast<size_t>(s.nq) * s.d);
  l.t_act = take(8 * static_cast<size_t>(s.I));
  l.t_part = take(8 * static_cast<size_t>(s.nkv) * kMegaSplitMax * s.rep * (s.d + 2));
  l.hist = take(sizeof(int) * static_cast<size_t>(s.B) * l.cap);
  l.slog = take(sizeof(float) * static_cast<size_t>(s.B) * s.V);
  l.sample_row = sample_row_bytes(s.V);
  l.sscr = take(kSampleBarBytes + static_cast<size_t>(s.B) * l.sample_row);
  {  // one fp32 scale per packed (pair- or tile-padded) row of every fp8 matrix
    const bool f8 = c.weight_dtype == K2_F8;
    auto rows = [&](int N, int kind) {
      const size_t pad = tiled_kind(kind) ? kQ4GroupRows : 2;
      return f8 ? sizeof(float) * pad * ((static_cast<size_t>(N) + pad - 1) / pad) : 0;
    };
    l.sqkv_layer = rows(s.qkv_n, 0);
    l.so_layer = rows(s.H, 1);
    l.sgu_layer = rows(2 * s.I, 2);
    l.sdown_layer = rows(s.H, 3);
    l.sqkv = take(l.sqkv_layer * s.L);
    l.so = take(l.so_layer * s.L);
    l.sgu = take(l.sgu_layer * s.L);
    l.sdown = take(l.sdown_layer * s.L);
    l.slm = take(rows(s.V, 4));
  }
  l.pchunk = (c.weight_dtype == K2_BF16 || c.weight_dtype == K2_F8 || c.weight_dtype == K2_Q4)
                 ? static_cast<int>(align_up(std::min(kPrefillChunk, s.ctx), 128))
                 : 0;
  {
    const size_t P = static_cast<size_t>(l.pchunk);
    const size_t kx = std::max(s.H, s.nq * s.d);
    l.px = take(P * s.H * 4);
    l.pxh = take(P * kx * 2);
    l.pxl = take(P * kx * 2);
    l.pah = take(P * s.I * 2);
    l.pal = take(P * s.I * 2);
    l.pqkv = take(P * s.qkv_n * 4);
    l.pq = take(P * s.nq * s.d * 4);
    l.plog = take(P > 0 ? static_cast<size_t>(s.B) * s.V * 4 : 0);  // batched-decode logits
    const size_t nv = P > 0 ? kSpecMax + 1 : 0;
    l.vlog = take(nv * s.V * 4);
    l.vids = take(sizeof(int) * (kSpecMax + 1));
    l.varg = take(sizeof(int) * (kSpecMax + 1));
    l.vpv = take(nv * kArgmaxPartsMax * 4);
    l.vpi = take(nv * kArgmaxPartsMax * 4);
  }
  const size_t scratch_end = o;
  // fp8 / int4: pair or tile units by GEMV kind (tiled_kind); else wb-byte
  // weights in 1024-byte units
  auto pbytes = [&](int N, int K, int kind) {
    return c.weight_dtype == K2_Q4   ? q4_packed_bytes(N, K, tiled_kind(kind))
           : c.weight_dtype == K2_F8 ? f8_packed_bytes(N, K, tiled_kind(kind))
                                     : packed_bytes(N, K, s.wb);
  };
  l.wqkv_layer = align_up(pbytes(s.qkv_n, s.H, 0), kAlign);
  l.wo_layer = align_up(pbytes(s.H, s.nq * s.d, 1), kAlign);
  l.wgu_layer = align_up(pbytes(2 * s.I, s.H, 2), kAlign);
  l.wdown_layer = align_up(pbytes(s.H, s.I, 3), kAlign);
  l.wqkv = take(l.wqkv_layer * s.L);
  l.wo = take(l.wo_layer * s.L);
  l.wgu = take(l.wgu_layer * s.L);
  l.wdown = take(l.wdown_layer * s.L);
  l.wlm = take(pbytes(s.V, s.H, 4));
  if (c.weight_dtype == K2_F8 && l.pchunk > 0) {  // bf16 copies of the fp8 codes for the prefill GEMMs
    l.tqkv_layer = align_up(packed_bytes(s.qkv_n, s.H, 2), kAlign);
    l.to_layer = align_up(packed_bytes(s.H, s.nq * s.d, 2), kAlign);
    l.tgu_layer = align_up(packed_bytes(2 * s.I, s.H, 2), kAlign);
    l.tdown_layer = align_up(packed_bytes(s.H, s.I, 2), kAlign);
    l.tqkv = take(l.tqkv_layer * s.L);
    l.to = take(l.to_layer * s.L);
    l.tgu = take(l.tgu_layer * s.L);
    l.tdown = take(l.tdown_layer * s.L);
  }
  if (c.weight_dtype == K2_BF16 && l.pchunk > 0) {  // two layers' weights as fp16, rebuilt per layer
    for (int b = 0; b < 2; ++b) {
      l.w16[b][0] = take(l.wqkv_layer);
      l.w16[b][1] = take(l.wo_layer);
      l.w16[b][2] = take(l.wgu_layer);
      l.w16[b][3] = take(l.wdown_layer);
    }
  }
  if (c.weight_dtype == K2_Q4 && l.pchunk > 0) {  // one layer's weights as bf16 hi / lo, rebuilt per layer
    const int Ns[4] = {s.qkv_n, s.H, 2 * s.I, s.H}, Ks[4] = {s.H, s.nq * s.d, s.H, s.I};
    for (int m = 0; m < 4; ++m) {
      l.dq_bytes[m] = align_up(packed_bytes(Ns[m], Ks[m], 2), kAlign);
      l.dq[m] = take(2 * l.dq_bytes[m]);
    }
  }
  l.repack_bytes = o - scratch_end;
  const size_t kv_start = o;
  l.kv_layer = align_up(static_cast<size_t>(s.B) * s.nkv * l.cap * s.d * s.kvb, kAlign);
  l.sc_layer = c.kv_dtype == K2_I8 ? align_up(static_cast<size_t>(s.B) * s.nkv * l.cap * 2, kAlign) : 0;
  l.kc = take(l.kv_layer * s.L);
  l.vc = take(l.kv_layer * s.L);
  l.ks = take(l.sc_layer * s.L);
  l.vs = take(l.sc_layer * s.L);
  l.kv_bytes = o - kv_start;
  l.total = o;
  return l;
}

std::string check_config(const k2_config* c) {
  if (!c) return "config is NULL";
  if (c->hidden <= 0 || c->n_layers <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
      c->intermediate <= 0 || c->norm_groups <= 0 || c->vocab <= 0 || c->max_context <= 0 || c->max_batch <= 0)
    return "every size in the config must be positive";
  if (c->hidden % c->norm_groups) return "hidden must be a multiple of norm_groups";
  if (c->n_heads % c->n_kv_heads) return "n_heads must be a multiple of n_kv_heads";
  if (c->head_dim % 2) return "head_dim must be even (split-half RoPE)";
  if (!(c->eps >= 0.f) || !(c->rope_theta > 0.f)) return "eps must be >= 0 and rope_theta > 0";
  if (c->weight_dtype != K2_F32 && c->weight_dtype != K2_BF16 && c->weight_dtype != K2_F8 &&
      c->weight_dtype != K2_Q4)
    return "weight_dtype must be K2_F32, K2_BF16, K2_F8 or K2_Q4";
  if (c->kv_dtype != K2_F32 && c->kv_dtype != K2_F16 && c->kv_dtype != K2_I8)
    return "kv_dtype must be K2_F32, K2_F16 or K2_I8";
  if (c->max_batch > 64) return "max_batch above 64 is not supported";
  if (c->max_context > (1 << 24)) return "max_context above 2^24 is not supported";
  if (!attn_supported(c->head_dim, c->n_heads / c->n_kv_heads, c->kv_dtype == K2_F32 ? 0 : c->kv_dtype))
    return "attention kernel not built for this head_dim / GQA ratio / kv dtype";
  return "";
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

// ---------------------------------------------------------------------------
// the context
// ---------------------------------------------------------------------------
struct k2_ctx {
  k2_config cfg;
  Sizes s;
  Layout lay;
  int sms = 0;
  uint8_t* ws = nullptr;
  // weights
  const void* embed = nullptr;
  const void* lm_head = nullptr;
  const void* final_norm = nullptr;
  std::vector<const void*> attn_norm, mlp_norm;
  // workspace pointers
  int* seq_len = nullptr;
  unsigned* guard = nullptr;
  unsigned* am_counter = nullptr;
  float2* rope = nullptr;
  float *resid = nullptr, *qkv = nullptr, *attn_out = nullptr, *act = nullptr, *attn_part = nullptr,
        *am_val = nullptr;
  int* am_idx = nullptr;
  int* hist = nullptr;   // [max_batch][cap] token ids of each sequence's cache rows
  float* slog = nullptr; // [max_batch][vocab] logits of a sampled step without caller logits
  // sampling (temperature 0: greedy)
  k2_sampling samp = {};
  bool sampling = false;
  std::vector<int> sample_cpr;  // CTAs per row of the sampler, by row count
  // plans
  PackedGemvArgs p_qkv = {}, p_o = {}, p_gu = {}, p_down = {}, p_lm = {};
  int grid_qkv = 0, grid_o = 0, grid_gu = 0, grid_down = 0, grid_lm = 0;
  AttnArgs p_attn = {};
  int attn_cluster_max = 1;  // largest launchable attention cluster
  int attn_resident = 1;     // attention CTAs resident on the whole GPU at once
  int force_splits = 0;
  // state
  std::vector<int> len;
  bool pdl = true;
  bool graph = false;
  // persistent batch-1 step
  bool mega_ok = false;
  bool use_mega = true;
  int mega_grid = 0;
  MegaArgs mega = {};
  KvMaps mega_maps = {};  // the persistent step's tensor maps of the caches (tensor-core attention)
  KvMaps pf_maps = {};    // the tcgen05 prefill attention's tensor maps of the caches (64-row boxes)
  bool pf_tc = false;     // fp16 cache of a supported shape: prefill attention on tcgen05
  bool use_pf_tc = true;  // option K2_OPT_PREFILL_ATTN
  int pf_split = 3;       // option K2_OPT_PREFILL_SPLIT (0 .. 3)
  bool pf_whole = true;   // option K2_OPT_PREFILL_GEMM
  std::vector<LayerPtrs> ltab;
  // tensor-core prefill: TMA tensor maps (weights per layer: qkv, o, gate/up,
  // down; activations: normed input, attention output, SwiGLU output, hi/lo)
  bool tc_ok = false;    // tensor-core prefill
  bool tc_full = false;  // and the paths that also need a bf16 lm_head (batched decode, speculation)
  bool use_tc = true;        // prefill
  bool use_tc_decode = true; // batched decode (batch >= 2)
  std::vector<std::array<uint8_t, kTcMapBytes>> tmw;  // 4 per layer
  std::array<uint8_t, kTcMapBytes> tm_xh{}, tm_xl{}, tm_oh{}, tm_ol{}, tm_ah{}, tm_al{}, tm_lm{};
  std::array<std::array<uint8_t, kTcMapBytes>, 4> tm_wlo{};  // int4: the weights' low halves
  // bf16 weights, fp16-operand prefill: the fp16 copies of layers of parity 0 / 1, converted on a
  // second stream while the previous layer computes (events: copy b ready, copy b read)
  std::array<std::array<std::array<uint8_t, kTcMapBytes>, 4>, 2> tm_w16{};
  bool w16_ok = false;
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_conv[2] = {}, ev_used[2] = {};
  ~k2_ctx() {
    if (side) cudaStreamDestroy(side);
    for (cudaEvent_t ev : {ev_fork, ev_join, ev_conv[0], ev_conv[1], ev_used[0], ev_used[1]})
      if (ev) cudaEventDestroy(ev);
  }
  // the same activation buffers in 16-token tiles (batched decode)
  std::array<uint8_t, kTcMapBytes> tb_xh{}, tb_xl{}, tb_oh{}, tb_ol{}, tb_ah{}, tb_al{};
  // and in 256-token tiles (fp16-operand prefill of long blocks: single activations)
  std::array<uint8_t, kTcMapBytes> tw_xh{}, tw_oh{}, tw_ah{};
  bool tw_ok = false;
  // fp16 caches: the tensor maps of each layer's K and V for the tensor-core decode attention
  std::vector<std::array<uint8_t, kTcMapBytes>> tm_k, tm_v;
  std::map<std::tuple<int, const void*, const void*, const void*, void*>, cudaGraphExec_t> graphs;
  std::map<std::tuple<int, int, void*>, cudaGraphExec_t> spec_graphs;  // (seq, ids verified (0: a plain step), stream)
  int spec_rows = 0;  // rows of logits the last speculative step left in the verification buffer
  unsigned long long poll_limit_ns = 1000000000ull;  // persistent step: waits for other CTAs' words (1 s)
  int stall_phase = -1;                              // persistent step: test option K2_OPT_STALL_PHASE
  // persistent step: L2 look-ahead per phase kind (two slots at the gate/up and
  // down phases measured fastest at context 4096: 1.934 against 1.990 ms per
  // token without; deeper look-ahead, or look-ahead at the attention phase, was
  // slower; quantized weights measured faster without it -- int4 1.85 against
  // 1.92 ms, fp8 1.66 against 1.71 ms -- so their default mask is 0)
  int l2_ahead = 2, l2_mask = 0x18;
  unsigned long long* trace = nullptr;               // persistent step: K2_OPT_TRACE buffer
  std::string err;
  // profiling: event pairs around the kernels of one step
  std::vector<cudaEvent_t> pev;

  void* wqkv(int l) const { return ws + lay.wqkv + lay.wqkv_layer * l; }
  void* wop(int l) const { return ws + lay.wo + lay.wo_layer * l; }
  void* wgu(int l) const { return ws + lay.wgu + lay.wgu_layer * l; }
  void* wdown(int l) const { return ws + lay.wdown + lay.wdown_layer * l; }
  void* wlm() const { return ws + lay.wlm; }
  // the bf16 weights of the prefill GEMMs (m: 0 QKV, 1 o_proj, 2 gate/up, 3 down) and,
  // for fp8 weights, their row scales
  bool f8() const { return cfg.weight_dtype == K2_F8; }
  bool q4() const { return cfg.weight_dtype == K2_Q4; }
  // int4: the dequantized halves of matrix m (rebuilt for every layer)
  void* dq_hi(int m) const { return ws + lay.dq[m]; }
  void* dq_lo(int m) const { return ws + lay.dq[m] + lay.dq_bytes[m]; }
  void* tcw(int l, int m) const {
    if (q4()) return dq_hi(m);
    if (!f8()) return m == 0 ? wqkv(l) : m == 1 ? wop(l) : m == 2 ? wgu(l) : wdown(l);
    const size_t base[4] = {lay.tqkv, lay.to, lay.tgu, lay.tdown};
    const size_t stride[4] = {lay.tqkv_layer, lay.to_layer, lay.tgu_layer, lay.tdown_layer};
    return ws + base[m] + stride[m] * l;
  }
  const float* tcs(int l, int m) const {
    if (!f8()) return nullptr;
    const size_t base[4] = {lay.sqkv, lay.so, lay.sgu, lay.sdown};
    const size_t stride[4] = {lay.sqkv_layer, lay.so_layer, lay.sgu_layer, lay.sdown_layer};
    return reinterpret_cast<const float*>(ws + base[m] + stride[m] * l);
  }
  void* kc(int l) const { return ws + lay.kc + lay.kv_layer * l; }
  void* vc(int l) const { return ws + lay.vc + lay.kv_layer * l; }
  void* ks(int l) const { return lay.sc_layer ? ws + lay.ks + lay.sc_layer * l : nullptr; }
  void* vs(int l) const { return lay.sc_layer ? ws + lay.vs + lay.sc_layer * l : nullptr; }

  k2_status fail(k2_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    err = buf;
    return st;
  }
  k2_status cuda_fail(cudaError_t e, const char* what) {
    return fail(K2_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  }
};

namespace {

// Key splits per (sequence, KV head): the count whose CTAs fill the last wave
// of resident CTAs best (a clearly fuller last wave wins; on a tie the fewer
// splits, which merge less), within the cluster limit and >= 8 keys per split.
int attn_splits(const k2_ctx* c, int batch) {
  if (c->force_splits > 0) return c->force_splits < c->attn_cluster_max ? c->force_splits : c->attn_cluster_max;
  const int items = c->s.nkv * batch;
  const int max_splits = std::max(1, std::min(c->attn_cluster_max, c->lay.cap / 8));
  int best = 1;
  double best_fill = -1.0;
  for (int n = 1; n <= max_splits; ++n) {
    const double waves = static_cast<double>(items) * n / c->attn_resident;
    const double fill = waves / std::ceil(waves);
    if (fill > best_fill + 0.02) {
      best = n;
      best_fill = fill;
    }
  }
  return best;
}

// Kernel launch recorder: plain launches, or (profiling) each launch between
// a pair of CUDA events; the events are read after the whole step has been
// queued, so the timings are device time, not host launch latency.
struct Launcher {
  k2_ctx* c;
  cudaStream_t s;
  bool pdl;
  bool profile = false;
  std::vector<int> classes;  // kernel class of each profiled launch
  cudaError_t err = cudaSuccess;

  template <typename F>
  void run(int cls, F&& f) {
    if (err != cudaSuccess) return;
    if (profile) {
      const size_t i = classes.size();
      while (c->pev.size() < 2 * (i + 1)) {
        cudaEvent_t e;
        if ((err = cudaEventCreate(&e))) return;
        c->pev.push_back(e);
      }
      if ((err = cudaEventRecord(c->pev[2 * i], s))) return;
      if ((err = f())) return;
      if ((err = cudaEventRecord(c->pev[2 * i + 1], s))) return;
      classes.push_back(cls);
    } else {
      err = f();
    }
  }
  // waits for the profiled launches and adds their device times per class
  cudaError_t collect(float* ms, int* launches) {
    if (err != cudaSuccess) return err;
    if (classes.empty()) return cudaSuccess;
    if ((err = cudaEventSynchronize(c->pev[2 * classes.size() - 1]))) return err;
    for (size_t i = 0; i < classes.size(); ++i) {
      float t = 0.f;
      if ((err = cudaEventElapsedTime(&t, c->pev[2 * i], c->pev[2 * i + 1]))) return err;
      ms[classes[i]] += t;
      launches[classes[i]] += 1;
    }
    return cudaSuccess;
  }
};

// One token of one sequence through the model with the batch-1 kernels.
//   tok: device token (null when x_in is given); x_in: caller's residual
//   stream (layers only); head: run final norm + lm_head + argmax (else only
//   advance the length).
// the decode attention of layer l reads an fp16 cache through its tensor maps
void attn_maps(const k2_ctx* c, AttnArgs& at, int l) {
  if (!c->tm_k.empty()) {
    at.map_k = c->tm_k[l].data();
    at.map_v = c->tm_v[l].data();
  }
}

void chain_b1(k2_ctx* c, Launcher& ln, int seq, const int* tok, float* x_in, int* next, float* logits, bool head) {
  const Sizes& s = c->s;
  const int wb = s.wb;
  float* x = x_in ? x_in : c->resid;
  cudaStream_t st = ln.s;
  const bool pdl = ln.pdl;
  if (!x_in)
    ln.run(K2_K_EMBED, [&] {
      return launch_embed(c->embed, wb, s.V, s.H, tok, 1, x, c->guard, c->hist + static_cast<size_t>(seq) * c->lay.cap,
                          c->lay.cap, c->seq_len + seq, st, pdl);
    });
  const int kvdt = c->cfg.kv_dtype == K2_F32 ? 0 : c->cfg.kv_dtype;
  const int splits = attn_splits(c, 1);
  for (int l = 0; l < s.L; ++l) {
    PackedGemvArgs q = c->p_qkv;
    q.Wp = c->wqkv(l);
    q.x = x;
    q.gain = c->attn_norm[l];
    q.out = c->qkv;
    q.seq = seq;
    ln.run(K2_K_QKV, [&] { return launch_packed_gemv(q, wb, EPI_QKV, c->grid_qkv, st, pdl); });

    AttnArgs at = c->p_attn;
    at.kc = at.kc_w = c->kc(l);
    at.vc = at.vc_w = c->vc(l);
    at.ks = c->ks(l);
    at.vs = c->vs(l);
    at.seq0 = seq;
    attn_maps(c, at, l);
    ln.run(K2_K_ATTN, [&] { return launch_attn(at, s.d, s.rep, kvdt, splits, 1, st, pdl); });

    PackedGemvArgs o = c->p_o;
    o.Wp = c->wop(l);
    o.x = c->attn_out;
    o.out = x;
    ln.run(K2_K_OPROJ, [&] { return launch_packed_gemv(o, wb, EPI_RESID, c->grid_o, st, pdl); });

    PackedGemvArgs gu = c->p_gu;
    gu.Wp = c->wgu(l);
    gu.x = x;
    gu.gain = c->mlp_norm[l];
    gu.out = c->act;
    ln.run(K2_K_GATEUP, [&] { return launch_packed_gemv(gu, wb, EPI_SWIGLU, c->grid_gu, st, pdl); });

    PackedGemvArgs dn = c->p_down;
    dn.Wp = c->wdown(l);
    dn.x = c->act;
    dn.out = x;
    ln.run(K2_K_DOWN, [&] { return launch_packed_gemv(dn, wb, EPI_RESID, c->grid_down, st, pdl); });
  }
  if (head) {
    PackedGemvArgs lm = c->p_lm;
    lm.x = x;
    lm.logits = logits;
    lm.next_token = next;
    lm.counter = c->am_counter + seq;
    lm.part_val = c->am_val + static_cast<size_t>(seq) * kArgmaxPartsMax;
    lm.part_idx = c->am_idx + static_cast<size_t>(seq) * kArgmaxPartsMax;
    lm.seq = seq;
    lm.advance = 1;
    ln.run(K2_K_LMHEAD, [&] { return launch_packed_gemv(lm, wb, EPI_ARGMAX, c->grid_lm, st, pdl); });
  } else {
    ln.run(K2_K_EMBED, [&] { return launch_advance(c->seq_len, seq, 1, st, pdl); });
  }
}

// One token of sequence seq: the persistent kernel when it can run, else the
// kernel chain.
void enqueue_token(k2_ctx* c, Launcher& ln, int seq, const int* tok, float* x_in, int* next, float* logits,
                   bool head) {
  if (c->mega_ok && c->use_mega) {
    MegaArgs m = c->mega;
    m.seq = seq;
    m.token_in = tok;
    m.token_out = next;
    m.logits = logits;
    m.x_ext = x_in;
    m.x_out = x_in ? x_in : c->resid + static_cast<size_t>(seq) * c->s.H;
    m.head = head ? 1 : 0;
    m.poll_limit_ns = c->poll_limit_ns;
    m.stall_phase = c->stall_phase;
    m.l2_ahead = c->l2_ahead;
    m.l2_mask = c->l2_mask;
    m.trace = c->trace;
    const int kvdt = c->cfg.kv_dtype == K2_F32 ? 0 : c->cfg.kv_dtype;
    cudaStream_t st = ln.s;
    ln.run(K2_K_STEP, [&] { return launch_mega(m, c->mega_maps, c->s.wf, c->s.d, c->s.rep, kvdt, c->mega_grid, st); });
  } else {
    chain_b1(c, ln, seq, tok, x_in, next, logits, head);
  }
}

cudaError_t decode_batched(k2_ctx* c, cudaStream_t st, const int* d_tokens, int B, int* d_next, float* d_logits);

// The sampler over `rows` rows of logits (k2_sample.cu), with the context's
// sampling parameters and scratch.
void enqueue_sample(k2_ctx* c, Launcher& ln, const float* logits, int rows, const int* seen, int seen_stride,
                    const int* seen_len, const int* pos, int first_seq, int* next) {
  SampleArgs a = {};
  a.logits = logits;
  a.ld = static_cast<size_t>(c->s.V);
  a.vocab = c->s.V;
  a.seen = c->samp.repetition_penalty != 1.0f ? seen : nullptr;
  a.seen_stride = seen_stride;
  a.seen_len = seen_len;
  a.counter = pos;
  a.first_seq = first_seq;
  a.next = next;
  a.temperature = c->samp.temperature;
  a.top_p = c->samp.top_p;
  a.min_p = c->samp.min_p;
  a.penalty = c->samp.repetition_penalty;
  a.top_k = c->samp.top_k;
  a.key0 = static_cast<uint32_t>(c->samp.seed);
  a.key1 = static_cast<uint32_t>(c->samp.seed >> 32);
  a.scratch = c->ws + c->lay.sscr;
  a.row_bytes = c->lay.sample_row;
  a.ctas_per_row = c->sample_cpr[rows];
  a.guard = c->guard;
  cudaStream_t st = ln.s;
  ln.run(K2_K_SAMPLE, [&] { return launch_sample(a, rows, st); });
}

void enqueue_decode(k2_ctx* c, Launcher& ln, const int* d_tokens, int batch, int* d_next, float* d_logits) {
  // a sampled step needs the logits: the caller's, else scratch
  float* lg = d_logits ? d_logits : (c->sampling ? c->slog : nullptr);
  if (batch >= 2 && batch <= 16 && c->tc_full && c->use_tc_decode) {
    ln.run(K2_K_STEP, [&] { return decode_batched(c, ln.s, d_tokens, batch, d_next, lg); });
  } else {
    for (int b = 0; b < batch; ++b)
      enqueue_token(c, ln, b, d_tokens + b, nullptr, d_next + b, lg ? lg + static_cast<size_t>(b) * c->s.V : nullptr,
                    true);
  }
  // the step advanced every length: it is the position each drawn token takes
  if (c->sampling) enqueue_sample(c, ln, lg, batch, c->hist, c->lay.cap, c->seq_len, c->seq_len, 0, d_next);
}

bool plan_all(k2_ctx* c) {
  const Sizes& s = c->s;
  // the kernel chain streams bf16 / fp32 weights; fp8 and int4 models run the
  // persistent step only (their chain plans, in bf16 terms, are never launched)
  const int wb = s.gb;
  PackedGemvArgs base = {};
  base.groups = s.G;
  base.eps = c->cfg.eps;
  base.rope = c->rope;
  base.cap = c->lay.cap;
  base.seq_len = c->seq_len;
  base.head_dim = s.d;
  base.n_rot_heads = s.nq + s.nkv;
  base.guard = c->guard;
  base.part_val = c->am_val;
  base.part_idx = c->am_idx;
  base.counter = c->am_counter;
  const void* dummy_gain = c->final_norm;  // any non-null: plans check the norm constraints
  c->p_qkv = base; c->p_qkv.N = s.qkv_n; c->p_qkv.K = s.H; c->p_qkv.gain = dummy_gain;
  c->p_o = base; c->p_o.N = s.H; c->p_o.K = s.nq * s.d;
  c->p_gu = base; c->p_gu.N = 2 * s.I; c->p_gu.K = s.H; c->p_gu.gain = dummy_gain;
  c->p_down = base; c->p_down.N = s.H; c->p_down.K = s.I;
  c->p_lm = base; c->p_lm.N = s.V; c->p_lm.K = s.H; c->p_lm.Wp = c->wlm(); c->p_lm.gain = c->final_norm;
  if (s.qkv_n % 2 || (2 * s.I) % 2) return false;  // pair epilogues
  // lm_head ends the step and no kernel overlaps it, so it takes a deeper ring
  if (!packed_plan(c->p_qkv, wb, kGemvSmem, 3) || !packed_plan(c->p_o, wb, kGemvSmem, 3) ||
      !packed_plan(c->p_gu, wb, kGemvSmem, 3) || !packed_plan(c->p_down, wb, kGemvSmem, 3) ||
      !packed_plan(c->p_lm, wb, kLmHeadSmem, kPackedMaxSlots))
    return false;
  c->p_o.gain = nullptr;
  c->p_down.gain = nullptr;
  c->grid_qkv = packed_grid(c->p_qkv.N, c->sms);
  c->grid_o = packed_grid(c->p_o.N, c->sms);
  c->grid_gu = packed_grid(c->p_gu.N, c->sms);
  c->grid_down = packed_grid(c->p_down.N, c->sms);
  c->grid_lm = packed_grid(c->p_lm.N, c->sms);

  AttnArgs& at = c->p_attn;
  at = {};
  at.cap = c->lay.cap;
  at.qkv = c->qkv;
  at.qkv_stride = s.qkv_n;
  at.nq = s.nq;
  at.nkv = s.nkv;
  at.seq_len = c->seq_len;
  at.out = c->attn_out;
  at.scale = static_cast<float>(1.0 / sqrt(static_cast<double>(s.d)));
  const int kvdt = c->cfg.kv_dtype == K2_F32 ? 0 : c->cfg.kv_dtype;
  at.slot_bytes = static_cast<uint32_t>(attn_slot_bytes(s.d, kvdt));
  at.guard = c->guard;
  return true;
}

// The persistent batch-1 step: supported shape, one CTA per SM, a device
// table of per-layer pointers.  Leaves mega_ok false when it cannot run.
cudaError_t plan_mega(k2_ctx* c, cudaStream_t st) {
  const Sizes& s = c->s;
  const int kvdt = c->cfg.kv_dtype == K2_F32 ? 0 : c->cfg.kv_dtype;
  c->mega_ok = false;
  if (!mega_supported(s.wf, s.d, s.rep, kvdt)) return cudaSuccess;
  const bool q4 = c->cfg.weight_dtype == K2_Q4, f8 = c->cfg.weight_dtype == K2_F8;
  const PackedGemvArgs* plans[5] = {&c->p_qkv, &c->p_o, &c->p_gu, &c->p_down, &c->p_lm};
  for (int kind = 0; kind < 5; ++kind) {
    const PackedGemvArgs* p = plans[kind];
    // the input vector, padded to whole chunks (int4: 64-weight blocks for
    // tiles, 512-weight chunks for pairs), fits its buffer (a gain phase: 4096 values)
    const int q4c = tiled_kind(kind) ? kQ4Block : kQ4Chunk;
    const size_t kp = q4 || (f8 && tiled_kind(kind)) ? static_cast<size_t>((p->K + q4c - 1) / q4c) * q4c
                                                     : p->x_bytes / 4;
    if (p->x_bytes > static_cast<uint32_t>(kMegaXBytes) || kp * 4 > static_cast<size_t>(kMegaXBytes)) return cudaSuccess;
    if (p->gain && kp > 4096) return cudaSuccess;
  }
  cudaError_t e = mega_init_attrs(s.wf, s.d, s.rep, kvdt);
  if (e != cudaSuccess) return e;
  int grid = mega_max_grid(s.wf, s.d, s.rep, kvdt);
  // every CTA must own rows of every layer GEMV (the dataflow waits rely on
  // it); fp8 and int4 rows of the tiled kinds are owned in 16-row tiles (8 pairs)
  auto rb = [&](int kind) { return (q4 || f8) && tiled_kind(kind) ? kQ4GroupRows / 2 : 1; };  // pairs per owner unit
  auto owned = [&](int N, int kind) { return ((N + 1) / 2 + rb(kind) - 1) / rb(kind); };
  grid = std::min(grid, std::min(owned(s.qkv_n, 0), std::min(owned(s.H, 1), owned(2 * s.I, 2))));
  if (grid < s.nkv) return cudaSuccess;
  // the QKV and residual epilogues keep their CTA's pairs in shared memory
  if ((owned(s.qkv_n, 0) + grid - 1) / grid * rb(0) > kMegaPairsMax ||
      (owned(s.H, 1) + grid - 1) / grid * rb(1) > kMegaPairsMax)
    return cudaSuccess;
  // inputs are polled in groups of four words; the gains are copied in 16-byte
  // pieces into the x buffer above a 16 KB input
  if (s.H % 8 || (s.nq * s.d) % 4 || s.I % 4) return cudaSuccess;
  if (static_cast<size_t>(s.H) * s.gb > static_cast<size_t>(kMegaGainBytes)) return cudaSuccess;
  if (s.d / 2 > 64) return cudaSuccess;  // the RoPE row of the position is kept in shared memory
  if (s.L > kMegaMaxLayers) return cudaSuccess;
  // tags carry the phase index in kMegaTagShift bits
  if (5 * s.L + 1 >= (1 << kMegaTagShift)) return cudaSuccess;
  int nsplit = grid / s.nkv;
  if (nsplit > kMegaSplitMax) nsplit = kMegaSplitMax;
  if (nsplit > c->lay.cap / 8) nsplit = c->lay.cap / 8;
  if (nsplit < 1) return cudaSuccess;
  c->ltab.resize(s.L);
  for (int l = 0; l < s.L; ++l) {
    LayerPtrs& t = c->ltab[l];
    t.wqkv = c->wqkv(l);
    t.wo = c->wop(l);
    t.wgu = c->wgu(l);
    t.wdown = c->wdown(l);
    t.attn_norm = c->attn_norm[l];
    t.mlp_norm = c->mlp_norm[l];
    t.kc = c->kc(l);
    t.vc = c->vc(l);
    t.ks = c->ks(l);
    t.vs = c->vs(l);
  }
  LayerPtrs* dtab = reinterpret_cast<LayerPtrs*>(c->ws + c->lay.ltab);
  e = cudaMemcpyAsync(dtab, c->ltab.data(), sizeof(LayerPtrs) * s.L, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  auto gplan = [&](const PackedGemvArgs& p, int kind) {  // packed units per row pair (int4 tiles: per tile)
    MegaGemv g;
    g.CT = (q4 || f8) && tiled_kind(kind) ? (p.K + kQ4Block - 1) / kQ4Block
           : q4                              ? (p.K + kQ4Chunk - 1) / kQ4Chunk
                                             : (p.K * s.wb + 511) / 512;
    return g;
  };
  MegaArgs& m = c->mega;
  m = {};
  m.layers = dtab;
  m.hist = c->hist;
  if (c->cfg.weight_dtype == K2_F8) {
    m.sc_qkv = reinterpret_cast<const float*>(c->ws + c->lay.sqkv);
    m.sc_o = reinterpret_cast<const float*>(c->ws + c->lay.so);
    m.sc_gu = reinterpret_cast<const float*>(c->ws + c->lay.sgu);
    m.sc_down = reinterpret_cast<const float*>(c->ws + c->lay.sdown);
    m.sc_lm = reinterpret_cast<const float*>(c->ws + c->lay.slm);
    m.ss_qkv = c->lay.sqkv_layer / sizeof(float);
    m.ss_o = c->lay.so_layer / sizeof(float);
    m.ss_gu = c->lay.sgu_layer / sizeof(float);
    m.ss_down = c->lay.sdown_layer / sizeof(float);
  }
  m.n_layers = s.L;
  m.w_qkv = static_cast<const uint8_t*>(c->wqkv(0));
  m.w_o = static_cast<const uint8_t*>(c->wop(0));
  m.w_gu = static_cast<const uint8_t*>(c->wgu(0));
  m.w_down = static_cast<const uint8_t*>(c->wdown(0));
  m.ws_qkv = c->lay.wqkv_layer;
  m.ws_o = c->lay.wo_layer;
  m.ws_gu = c->lay.wgu_layer;
  m.ws_down = c->lay.wdown_layer;
  m.kc = static_cast<uint8_t*>(c->kc(0));
  m.vc = static_cast<uint8_t*>(c->vc(0));
  m.ks = static_cast<uint8_t*>(c->ks(0));
  m.vs = static_cast<uint8_t*>(c->vs(0));
  m.s_kv = c->lay.kv_layer;
  m.s_sc = c->lay.sc_layer;
  m.embed = c->embed;
  m.lm_head = c->wlm();
  m.final_norm = c->final_norm;
  m.hidden = s.H;
  m.vocab = s.V;
  m.nq = s.nq;
  m.nkv = s.nkv;
  m.groups = s.G;
  m.inter = s.I;
  m.eps = c->cfg.eps;
  m.scale = static_cast<float>(1.0 / sqrt(static_cast<double>(s.d)));
  m.g_qkv = gplan(c->p_qkv, 0);
  m.g_o = gplan(c->p_o, 1);
  m.g_gu = gplan(c->p_gu, 2);
  m.g_down = gplan(c->p_down, 3);
  m.g_lm = gplan(c->p_lm, 4);
  m.cap = c->lay.cap;
  m.nsplit = nsplit;
  m.rope = c->rope;
  m.seq_len = c->seq_len;
  m.x_out = c->resid;
  m.t_resid = reinterpret_cast<unsigned long long*>(c->ws + c->lay.t_resid);
  m.t_qkv = reinterpret_cast<unsigned long long*>(c->ws + c->lay.t_qkv);
  m.t_attn = reinterpret_cast<unsigned long long*>(c->ws + c->lay.t_attn);
  m.t_act = reinterpret_cast<unsigned long long*>(c->ws + c->lay.t_act);
  m.t_part = reinterpret_cast<unsigned long long*>(c->ws + c->lay.t_part);
  m.am_val = c->am_val;
  m.am_idx = c->am_idx;
  m.end_count = reinterpret_cast<unsigned*>(c->ws + c->lay.msync);
  m.epoch = m.end_count + 1;
  m.guard = c->guard;
  if (mega_tc_attention(s.d, kvdt)) {
    const long long rows = static_cast<long long>(s.B) * s.nkv * c->lay.cap;
    if (!attn_encode_kv_layers(&c->mega_maps.k, c->kc(0), rows, s.d, s.L, c->lay.kv_layer, kMegaTK) ||
        !attn_encode_kv_layers(&c->mega_maps.v, c->vc(0), rows, s.d, s.L, c->lay.kv_layer, kMegaTK))
      return cudaSuccess;  // no tensor maps: the persistent step stays off (mega_ok false)
  }
  c->mega_grid = grid;
  c->mega_ok = true;
  return cudaSuccess;
}

// Tensor maps of the tensor-core prefill (bf16 weights, fp8 weights through
// bf16 copies of their codes, or int4 weights through one layer at a time
// dequantized into bf16 halves; a supported attention shape).  Leaves tc_ok
// false when it cannot run; tc_full (batched decode, speculation: a bf16
// lm_head) only for bf16 weights.
cudaError_t plan_tc_prefill(k2_ctx* c) {
  const Sizes& s = c->s;
  c->tc_ok = c->tc_full = false;
  if (c->lay.pchunk <= 0 || s.gb != 2 || !prefill_attn_supported(s.d, s.rep)) return cudaSuccess;
  if (s.H % 8 || (s.nq * s.d) % 8 || s.I % 8) return cudaSuccess;
  cudaError_t e = prefill_init_attrs();
  if (e != cudaSuccess) return e;
  c->tmw.resize(4 * static_cast<size_t>(s.L));
  for (int l = 0; l < s.L; ++l) {
    if (!tc_encode_weight(c->tmw[4 * l].data(), c->tcw(l, 0), s.qkv_n, s.H) ||
        !tc_encode_weight(c->tmw[4 * l + 1].data(), c->tcw(l, 1), s.H, s.nq * s.d) ||
        !tc_encode_weight(c->tmw[4 * l + 2].data(), c->tcw(l, 2), 2 * s.I, s.H) ||
        !tc_encode_weight(c->tmw[4 * l + 3].data(), c->tcw(l, 3), s.H, s.I))
      return cudaSuccess;
  }
  if (c->q4()) {
    const int Ns[4] = {s.qkv_n, s.H, 2 * s.I, s.H}, Ks[4] = {s.H, s.nq * s.d, s.H, s.I};
    for (int m = 0; m < 4; ++m)
      if (!tc_encode_weight(c->tm_wlo[m].data(), c->dq_lo(m), Ns[m], Ks[m])) return cudaSuccess;
  }
  if (c->cfg.weight_dtype == K2_BF16) {  // the tensor maps copy bytes: a bf16 map reads the fp16 copy as well
    const int Ns[4] = {s.qkv_n, s.H, 2 * s.I, s.H}, Ks[4] = {s.H, s.nq * s.d, s.H, s.I};
    bool ok = true;
    for (int b = 0; b < 2; ++b)
      for (int m = 0; m < 4; ++m)
        ok = ok && tc_encode_weight(c->tm_w16[b][m].data(), c->ws + c->lay.w16[b][m], Ns[m], Ks[m]);
    ok = ok && cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking) == cudaSuccess;
    for (cudaEvent_t* ev : {&c->ev_fork, &c->ev_join, &c->ev_conv[0], &c->ev_conv[1], &c->ev_used[0], &c->ev_used[1]})
      ok = ok && cudaEventCreateWithFlags(ev, cudaEventDisableTiming) == cudaSuccess;
    c->w16_ok = ok;
  }
  const int P = c->lay.pchunk;
  c->tw_ok = P > 512 && tc_encode_act(c->tw_xh.data(), c->ws + c->lay.pxh, P, s.H, 256) &&
             tc_encode_act(c->tw_oh.data(), c->ws + c->lay.pxh, P, s.nq * s.d, 256) &&
             tc_encode_act(c->tw_ah.data(), c->ws + c->lay.pah, P, s.I, 256);
  bool ok = true;
  for (int tt : {128, 16}) {
    ok = ok && tc_encode_act((tt == 128 ? c->tm_xh : c->tb_xh).data(), c->ws + c->lay.pxh, P, s.H, tt) &&
         tc_encode_act((tt == 128 ? c->tm_xl : c->tb_xl).data(), c->ws + c->lay.pxl, P, s.H, tt) &&
         tc_encode_act((tt == 128 ? c->tm_oh : c->tb_oh).data(), c->ws + c->lay.pxh, P, s.nq * s.d, tt) &&
         tc_encode_act((tt == 128 ? c->tm_ol : c->tb_ol).data(), c->ws + c->lay.pxl, P, s.nq * s.d, tt) &&
         tc_encode_act((tt == 128 ? c->tm_ah : c->tb_ah).data(), c->ws + c->lay.pah, P, s.I, tt) &&
         tc_encode_act((tt == 128 ? c->tm_al : c->tb_al).data(), c->ws + c->lay.pal, P, s.I, tt);
  }
  // the batched decode keeps the gate/up output of 16 tokens in the QKV buffer
  if (16 * 2 * static_cast<size_t>(s.I) > static_cast<size_t>(P) * s.qkv_n) return cudaSuccess;
  if (!ok) return cudaSuccess;
  c->tc_ok = true;
  c->tc_full = !quantized(c->cfg.weight_dtype) && tc_encode_weight(c->tm_lm.data(), c->wlm(), s.V, s.H);
  return cudaSuccess;
}

// One block of n <= pchunk prompt tokens of sequence seq at positions
// pos0 .. pos0+n-1 through every layer; the residual of its last token is left
// in pX[n-1].
// d_pos0 (nullable): the block's first position read on the device (a graph
// replayed at any position), else pos0
cudaError_t prefill_block(k2_ctx* c, int seq, const int* d_tokens, int n, int pos0, cudaStream_t st,
                          const int* d_pos0 = nullptr) {
  const Sizes& s = c->s;
  float* X = reinterpret_cast<float*>(c->ws + c->lay.px);
  auto* xh = reinterpret_cast<__nv_bfloat16*>(c->ws + c->lay.pxh);
  auto* xl = reinterpret_cast<__nv_bfloat16*>(c->ws + c->lay.pxl);
  auto* ah = reinterpret_cast<__nv_bfloat16*>(c->ws + c->lay.pah);
  auto* al = reinterpret_cast<__nv_bfloat16*>(c->ws + c->lay.pal);
  float* qkv = reinterpret_cast<float*>(c->ws + c->lay.pqkv);
  float* Q = reinterpret_cast<float*>(c->ws + c->lay.pq);
  const int kvdt = c->cfg.kv_dtype == K2_F32 ? 0 : c->cfg.kv_dtype;
  const size_t head_row0 = static_cast<size_t>(seq) * s.nkv * c->lay.cap;
  const float scale = static_cast<float>(1.0 / sqrt(static_cast<double>(s.d)));
  // rs: the weight rows' scales (fp8 codes), else null
  // int4: before its GEMM, each matrix of the layer is dequantized into bf16
  // halves (c->dq_*), and the GEMM adds the low halves' products
  const bool q4 = c->q4();
  // a block of at most 16 tokens (a speculative verification) streams every
  // weight matrix with the stream-K kernel over 16-token tiles, one CTA per
  // SM: the 128-token tiles would leave most SMs idle (int4 weights keep the
  // 128-token tiles, the only ones with a low-half weight operand)
  const bool small = n <= 16 && !q4;
  // fp16 operands (option K2_OPT_PREFILL_SPLIT = 3: bf16 weights, fp16 caches on
  // the tcgen05 attention, blocks over 16 tokens): each matrix of the layer is
  // converted to fp16 (exact in fp16's normal range) before its GEMM, and the
  // activations enter as single fp16; elsewhere 3 acts as 1
  const bool f16 =
      c->pf_split == 3 && c->cfg.weight_dtype == K2_BF16 && !small && c->pf_tc && c->use_pf_tc && c->w16_ok;
  const int mode = f16 ? 3 : c->pf_split == 3 ? 1 : c->pf_split;
  // long fp16 blocks: 256-token tiles (each SM receives 1.5x the bytes of a
  // 128-token tile per K step for twice its MMAs)
  const bool wide = f16 && n > 512 && c->pf_whole && c->tw_ok;
  auto wmap = [&](int l, int m) -> const void* {
    return f16 ? c->tm_w16[l & 1][m].data() : c->tmw[4 * l + m].data();
  };
  // fp16: layer l's four matrices into copy l & 1 on the second stream
  auto convert_layer = [&](int l) {
    const void* srcs[4] = {c->wqkv(l), c->wop(l), c->wgu(l), c->wdown(l)};
    const int Ns[4] = {s.qkv_n, s.H, 2 * s.I, s.H}, Ks[4] = {s.H, s.nq * s.d, s.H, s.I};
    cudaError_t e = cudaSuccess;
    for (int m = 0; m < 4 && !e; ++m)
      e = launch_bf16_to_f16(reinterpret_cast<__half*>(c->ws + c->lay.w16[l & 1][m]),
                             static_cast<const __nv_bfloat16*>(srcs[m]), packed_bytes(Ns[m], Ks[m], 2) / 2, c->guard,
                             c->side);
    return e ? e : cudaEventRecord(c->ev_conv[l & 1], c->side);
  };
  const void* wlo = nullptr;
  auto dequant = [&](int l, int m) {
    if (f16) return cudaSuccess;  // converted ahead on the second stream
    if (!q4) {
      wlo = nullptr;
      return cudaSuccess;
    }
    wlo = c->tm_wlo[m].data();
    const void* srcs[4] = {c->wqkv(l), c->wop(l), c->wgu(l), c->wdown(l)};
    const int Ns[4] = {s.qkv_n, s.H, 2 * s.I, s.H}, Ks[4] = {s.H, s.nq * s.d, s.H, s.I};
    return launch_q4_dequant(c->dq_hi(m), c->dq_lo(m), static_cast<const uint8_t*>(srcs[m]), Ns[m], Ks[m],
                             tiled_kind(m), st);
  };
  auto gemm = [&](const void* mw, const float* rs, const void* mh, const void* ml, int N, int K, int mode, float* out,
                  __nv_bfloat16* oh, __nv_bfloat16* ol, int ldo) {
    TcGemmArgs g = {};
    g.N = N;
    g.K = K;
    g.T = n;
    g.ksteps = 4 * ((K + 255) / 256);
    g.mode = mode;
    g.ldo = ldo;
    g.tile_tokens = wide ? 256 : 128;
    g.splits = 1;
    g.out = out;
    g.out_hi = oh;
    g.out_lo = ol;
    g.guard = c->guard;
    g.row_scale = rs;
    g.f16 = f16 ? 1 : 0;
    if (!c->pf_whole) return launch_tc_gemm(mw, wlo, mh, ml, g, st);
    g.whole = 1;
    // programmatic dependent launch: the GEMM requests its first weight stages
    // while the kernel before it (a norm, which lets dependents start at once)
    // still runs, and waits for it before reading the activations
    return launch_tc_gemm_sk(mw, wlo, mh, ml, g, c->sms, st, c->pdl);
  };
  const int tt = small ? 16 : 128;
  auto gemm_sk = [&](const void* mw, const float* rs, const void* mh, const void* ml, int N, int K, int mode, float* out,
                     int ldo) {
    TcGemmArgs g = {};
    g.N = N;
    g.K = K;
    g.T = n;
    g.ksteps = 4 * ((K + 255) / 256);
    g.mode = mode;
    g.ldo = ldo;
    g.tile_tokens = wide ? 256 : tt;
    g.splits = 1;
    g.out = out;
    g.guard = c->guard;
    g.row_scale = rs;
    g.f16 = f16 ? 1 : 0;
    cudaError_t e = cudaSuccess;
    if (mode == TC_STORE) e = cudaMemsetAsync(out, 0, sizeof(float) * static_cast<size_t>(n) * ldo, st);
    if (!e) e = launch_tc_gemm_sk(mw, wlo, mh, ml, g, c->sms, st, c->pdl && !small);
    return e;
  };
  // without the split (blocks over 16 tokens only) the low-half maps are null:
  // the GEMMs read the high halves alone
  // int4: the low-half weight MMA needs the activations' halves
  const bool split = !f16 && (small || mode != 0 || q4);
  const bool attn_split = small || mode == 1;  // 2, 3: the attention's Q and P single
  const void* m_xh = small ? c->tb_xh.data() : wide ? c->tw_xh.data() : c->tm_xh.data();
  const void* m_xl = small ? c->tb_xl.data() : split ? c->tm_xl.data() : nullptr;
  const void* m_oh = small ? c->tb_oh.data() : wide ? c->tw_oh.data() : c->tm_oh.data();
  const void* m_ol = small ? c->tb_ol.data() : split ? c->tm_ol.data() : nullptr;
  const void* m_ah = small ? c->tb_ah.data() : wide ? c->tw_ah.data() : c->tm_ah.data();
  const void* m_al = small ? c->tb_al.data() : split ? c->tm_al.data() : nullptr;
  cudaError_t e = launch_embed_rows(d_tokens, n, c->embed, s.gb, X, s.H, s.V, c->guard,
                                    c->hist + static_cast<size_t>(seq) * c->lay.cap, 0, nullptr, pos0, d_pos0, st);
  if (f16 && !e) {
    // the second stream starts after the work already on st (an earlier
    // prefill may still read the copies) and converts the first two layers
    e = cudaEventRecord(c->ev_fork, st);
    if (!e) e = cudaStreamWaitEvent(c->side, c->ev_fork, 0);
    for (int l = 0; l < std::min(2, s.L) && !e; ++l) e = convert_layer(l);
  }
  for (int l = 0; l < s.L && !e; ++l) {
    if (f16 && !e) e = cudaStreamWaitEvent(st, c->ev_conv[l & 1], 0);
    if (!e)
      e = launch_norm_rows(X, n, c->attn_norm[l], s.gb, xh, xl, s.H, s.G, c->cfg.eps, st, false, nullptr, 0, nullptr,
                           f16, c->guard);
    if (!e) e = dequant(l, 0);
    if (!e)
      e = small ? gemm_sk(wmap(l, 0), c->tcs(l, 0), m_xh, m_xl, s.qkv_n, s.H, TC_STORE, qkv, s.qkv_n)
                : gemm(wmap(l, 0), c->tcs(l, 0), m_xh, m_xl, s.qkv_n, s.H, TC_STORE, qkv, nullptr, nullptr, s.qkv_n);
    if (!e)
      e = launch_rope_append(qkv, Q, c->rope, kvdt, c->kc(l), c->vc(l), c->ks(l), c->vs(l), n, s.nq, s.nkv, s.d,
                             pos0, d_pos0, head_row0, c->lay.cap, st, c->pdl);
    if (!e && small) {
      // few queries over a long history: the decode attention in block mode
      // splits every query's keys over a cluster of CTAs
      AttnArgs at = c->p_attn;
      at.kc = at.kc_w = c->kc(l);
      at.vc = at.vc_w = c->vc(l);
      at.ks = c->ks(l);
      at.vs = c->vs(l);
      at.qkv = Q;
      at.qkv_stride = s.nq * s.d;
      at.seq0 = 0;
      at.block_mode = 1;
      at.block_seq = seq;
      at.pos_base = pos0;
      at.pos_base_dev = d_pos0;
      at.out = nullptr;  // the merged output goes straight to the o_proj GEMM's bf16 halves
      at.out_hi = xh;
      at.out_lo = xl;
      attn_maps(c, at, l);
      e = launch_attn(at, s.d, s.rep, kvdt, attn_splits(c, n), n, st, false);
    } else if (!e && c->pf_tc && c->use_pf_tc) {
      PrefillAttnArgs pa = {};
      pa.Q = Q;
      pa.oh = xh;
      pa.ol = split ? xl : nullptr;
      pa.split = attn_split ? 1 : 0;
      pa.f16out = f16 ? 1 : 0;
      pa.n = n;
      pa.nq = s.nq;
      pa.nkv = s.nkv;
      pa.pos0 = pos0;
      pa.head_row0 = static_cast<int>(head_row0);
      pa.cap = c->lay.cap;
      pa.layer = l;
      pa.scale = scale;
      pa.guard = c->guard;
      e = launch_prefill_attn_tc(c->pf_maps, pa, s.d, s.rep, st);
    } else if (!e) {
      e = launch_prefill_attn(Q, kvdt, c->kc(l), c->vc(l), c->ks(l), c->vs(l), xh, xl, n, s.nq, s.nkv, s.d, pos0,
                              head_row0, c->lay.cap, scale, st);
    }
    // o_proj and down have few row tiles: stream-K over one CTA per SM
    if (!e) e = dequant(l, 1);
    if (!e) e = gemm_sk(wmap(l, 1), c->tcs(l, 1), m_oh, m_ol, s.H, s.nq * s.d, TC_RESID, X, s.H);
    if (!e)
      e = launch_norm_rows(X, n, c->mlp_norm[l], s.gb, xh, xl, s.H, s.G, c->cfg.eps, st, false, nullptr, 0, nullptr,
                           f16, c->guard);
    if (!e) e = dequant(l, 2);
    if (!e) {
      if (small) {  // gate/up rows to fp32 (the QKV buffer is free by now), then SwiGLU rows
        e = gemm_sk(wmap(l, 2), c->tcs(l, 2), m_xh, m_xl, 2 * s.I, s.H, TC_STORE, qkv, 2 * s.I);
        if (!e) e = launch_swiglu_rows(qkv, ah, al, n, s.I, st);
      } else {
        e = gemm(wmap(l, 2), c->tcs(l, 2), m_xh, m_xl, 2 * s.I, s.H, TC_SWIGLU, nullptr, ah, split ? al : nullptr,
                 s.I);
      }
    }
    if (!e) e = dequant(l, 3);
    if (!e) e = gemm_sk(wmap(l, 3), c->tcs(l, 3), m_ah, m_al, s.H, s.I, TC_RESID, X, s.H);
    if (f16 && !e && l + 2 < s.L) {  // copy l & 1 is free once layer l's GEMMs have run: layer l + 2 goes there
      e = cudaEventRecord(c->ev_used[l & 1], st);
      if (!e) e = cudaStreamWaitEvent(c->side, c->ev_used[l & 1], 0);
      if (!e) e = convert_layer(l + 2);
    }
  }
  if (f16) {  // st waits for everything issued on the second stream (a failed call included)
    cudaError_t j = cudaEventRecord(c->ev_join, c->side);
    if (!j) j = cudaStreamWaitEvent(st, c->ev_join, 0);
    if (!e) e = j;
  }
  return e;
}

// Decode of tokens d_tokens[0..B) of sequences 0..B-1 (B >= 2) with the
// weights read once for all of them: tensor-core GEMMs with N = B tokens
// (split-K where a GEMM has few row tiles), the batched attention kernel, and
// a row-wise argmax.  Leaves each sequence's residual in its hidden view.
cudaError_t decode_batched(k2_ctx* c, cudaStream_t st, const int* d_tokens, int B, int* d_next, float* d_logits) {
  const Sizes& s = c->s;
  float* X = reinterpret_cast<float*>(c->ws + c->lay.px);
  auto* xh = reinterpret_cast<__nv_bfloat16*>(c->ws + c->lay.pxh);
  auto* xl = reinterpret_cast<__nv_bfloat16*>(c->ws + c->lay.pxl);
  auto* ah = reinterpret_cast<__nv_bfloat16*>(c->ws + c->lay.pah);
  auto* al = reinterpret_cast<__nv_bfloat16*>(c->ws + c->lay.pal);
  float* gout = reinterpret_cast<float*>(c->ws + c->lay.pqkv);  // QKV, then gate/up GEMM output
  float* logits = d_logits ? d_logits : reinterpret_cast<float*>(c->ws + c->lay.plog);
  const int kvdt = c->cfg.kv_dtype == K2_F32 ? 0 : c->cfg.kv_dtype;
  // Every launch of the step uses programmatic dependent launch: a kernel may
  // start while its predecessor drains and waits for it (griddepcontrol.wait)
  // before reading its output; the stream-K GEMMs request their first weight
  // stages before that wait.  The GEMMs add their partial sums with fp32 atomics
  // into `out`: a target that is not the residual stream is cleared by the norm
  // kernel in front of the GEMM (a memset node would break the chain).
  auto gemm = [&](const void* mw, const void* mh, const void* ml, int N, int K, int mode, float* out, int ldo) {
    TcGemmArgs g = {};
    g.N = N;
    g.K = K;
    g.T = B;
    g.ksteps = 4 * ((K + 255) / 256);
    g.mode = mode;
    g.ldo = ldo;
    g.tile_tokens = 16;
    g.splits = 1;
    g.out = out;
    g.guard = c->guard;
    return launch_tc_gemm_sk(mw, nullptr, mh, ml, g, c->sms, st, true);
  };
  // the final norm clears the logits unless the caller's buffer is not 16-byte aligned
  const bool lg_aligned = reinterpret_cast<uintptr_t>(logits) % 16 == 0 && (static_cast<size_t>(B) * s.V) % 4 == 0;
  const int asplits = attn_splits(c, B);
  cudaError_t e = launch_embed_rows(d_tokens, B, c->embed, s.wb, X, s.H, s.V, c->guard, c->hist, c->lay.cap,
                                    c->seq_len, 0, nullptr, st, true);
  for (int l = 0; l < s.L && !e; ++l) {
    if (!e)
      e = launch_norm_rows(X, B, c->attn_norm[l], s.wb, xh, xl, s.H, s.G, c->cfg.eps, st, true, gout,
                           static_cast<size_t>(B) * s.qkv_n);
    if (!e) e = gemm(c->tmw[4 * l].data(), c->tb_xh.data(), c->tb_xl.data(), s.qkv_n, s.H, TC_STORE, gout, s.qkv_n);
    if (!e) {
      // the attention reads the QKV GEMM's packed rows and rotates q and k itself
      AttnArgs at = c->p_attn;
      at.qkv = gout;
      at.qkv_stride = s.qkv_n;
      at.rope = c->rope;
      at.kc = at.kc_w = c->kc(l);
      at.vc = at.vc_w = c->vc(l);
      at.ks = c->ks(l);
      at.vs = c->vs(l);
      at.seq0 = 0;
      at.out = nullptr;  // the merged output goes straight to the o_proj GEMM's bf16 halves
      at.out_hi = xh;
      at.out_lo = xl;
      attn_maps(c, at, l);
      e = launch_attn(at, s.d, s.rep, kvdt, asplits, B, st, true);
    }
    if (!e) e = gemm(c->tmw[4 * l + 1].data(), c->tb_oh.data(), c->tb_ol.data(), s.H, s.nq * s.d, TC_RESID, X, s.H);
    if (!e)
      e = launch_norm_rows(X, B, c->mlp_norm[l], s.wb, xh, xl, s.H, s.G, c->cfg.eps, st, true, gout,
                           static_cast<size_t>(B) * 2 * s.I);
    if (!e)
      e = gemm(c->tmw[4 * l + 2].data(), c->tb_xh.data(), c->tb_xl.data(), 2 * s.I, s.H, TC_STORE, gout, 2 * s.I);
    if (!e) e = launch_swiglu_rows(gout, ah, al, B, s.I, st, true);
    if (!e) e = gemm(c->tmw[4 * l + 3].data(), c->tb_ah.data(), c->tb_al.data(), s.H, s.I, TC_RESID, X, s.H);
  }
  // the final norm also leaves the residual in the hidden view
  if (!e && !lg_aligned) e = cudaMemsetAsync(logits, 0, sizeof(float) * static_cast<size_t>(B) * s.V, st);
  if (!e)
    e = launch_norm_rows(X, B, c->final_norm, s.wb, xh, xl, s.H, s.G, c->cfg.eps, st, true,
                         lg_aligned ? logits : nullptr, lg_aligned ? static_cast<size_t>(B) * s.V : 0, c->resid);
  if (!e) e = gemm(c->tm_lm.data(), c->tb_xh.data(), c->tb_xl.data(), s.V, s.H, TC_STORE, logits, s.V);
  if (!e) e = launch_argmax_rows(logits, B, s.V, d_next, c->am_val, c->am_idx, kArgmaxPartsMax, c->guard, st, true);
  if (!e) e = launch_advance(c->seq_len, 0, B, st, true);
  return e;
}

// The whole prompt through tensor-core blocks, then the greedy head on the
// last token's residual (which is also left in the hidden view of seq).
cudaError_t prefill_tc(k2_ctx* c, int seq, const int* d_tokens, int n, int* d_next, float* d_logits,
                       cudaStream_t st) {
  const Sizes& s = c->s;
  const int P = c->lay.pchunk;
  cudaError_t e = cudaSuccess;
  int last = 0;
  // fp8 / int4 weights: the lm_head exists only in their packed form, so the
  // last token takes the persistent step (which ends in the lm_head and argmax)
  const bool quant = quantized(c->cfg.weight_dtype);
  const int nb = quant ? n - 1 : n;
  for (int b0 = 0; b0 < nb && !e; b0 += P) {
    last = std::min(P, nb - b0);
    e = prefill_block(c, seq, d_tokens + b0, last, c->len[seq] + b0, st);
  }
  if (e) return e;
  if (quant) {
    if ((e = launch_advance_by(c->seq_len, seq, nb, st)) != cudaSuccess) return e;
    Launcher ln{c, st, false};
    enqueue_token(c, ln, seq, d_tokens + nb, nullptr, d_next, d_logits, true);
    return ln.err;
  }
  float* xrow = c->resid + static_cast<size_t>(seq) * s.H;
  e = cudaMemcpyAsync(xrow, c->ws + c->lay.px + static_cast<size_t>(last - 1) * s.H * 4, sizeof(float) * s.H,
                      cudaMemcpyDeviceToDevice, st);
  if (e) return e;
  PackedGemvArgs lm = c->p_lm;
  lm.x = xrow;
  lm.logits = d_logits;
  lm.next_token = d_next;
  lm.counter = c->am_counter + seq;
  lm.part_val = c->am_val + static_cast<size_t>(seq) * kArgmaxPartsMax;
  lm.part_idx = c->am_idx + static_cast<size_t>(seq) * kArgmaxPartsMax;
  lm.seq = seq;
  lm.advance = 0;
  e = launch_packed_gemv(lm, s.wb, EPI_ARGMAX, c->grid_lm, st, false);
  if (e) return e;
  return launch_advance_by(c->seq_len, seq, n, st);
}

// Appends the n ids at d_tokens (the next input and the drafts) to sequence
// seq in one tensor-core pass and writes the greedy id after every one of
// them (kimi-k3-in-c k3_run.c, --spec: batched greedy verification; the
// logits of every position).  The device length is left to the caller.
cudaError_t verify_block(k2_ctx* c, int seq, const int* d_tokens, int n, int* d_argmax, cudaStream_t st) {
  const Sizes& s = c->s;
  cudaError_t e = prefill_block(c, seq, d_tokens, n, c->len[seq], st, c->seq_len + seq);
  float* X = reinterpret_cast<float*>(c->ws + c->lay.px);
  auto* xh = reinterpret_cast<__nv_bfloat16*>(c->ws + c->lay.pxh);
  auto* xl = reinterpret_cast<__nv_bfloat16*>(c->ws + c->lay.pxl);
  float* logits = reinterpret_cast<float*>(c->ws + c->lay.vlog);
  if (!e) e = launch_norm_rows(X, n, c->final_norm, s.gb, xh, xl, s.H, s.G, c->cfg.eps, st);
  if (!e) e = cudaMemsetAsync(logits, 0, sizeof(float) * static_cast<size_t>(n) * s.V, st);
  if (!e) {
    TcGemmArgs g = {};
    g.N = s.V;
    g.K = s.H;
    g.T = n;
    g.ksteps = 4 * ((s.H + 255) / 256);
    g.mode = TC_STORE;
    g.ldo = s.V;
    g.tile_tokens = 16;
    g.splits = 1;
    g.out = logits;
    g.guard = c->guard;
    e = launch_tc_gemm_sk(c->tm_lm.data(), nullptr, c->tb_xh.data(), c->tb_xl.data(), g, c->sms, st);
  }
  if (!e)
    e = launch_argmax_rows(logits, n, s.V, d_argmax, reinterpret_cast<float*>(c->ws + c->lay.vpv),
                           reinterpret_cast<int*>(c->ws + c->lay.vpi), kArgmaxPartsMax, c->guard, st);
  return e;
}

k2_status validate_weights(k2_ctx* c, const k2_weights* w) {
  auto ok = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % 16) == 0; };
  if (!w) return c->fail(K2_ERR_ARG, "weights is NULL");
  if (!ok(w->embed) || !ok(w->lm_head) || !ok(w->final_norm))
    return c->fail(K2_ERR_ARG, "embed / lm_head / final_norm must be non-null 16-byte aligned device pointers");
  const void* const* arrs[] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->mlp_norm, w->w_gate, w->w_up, w->w_down};
  const char* names[] = {"attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down"};
  for (int i = 0; i < 9; ++i) {
    if (!arrs[i]) return c->fail(K2_ERR_ARG, "weights.%s is NULL", names[i]);
    for (int l = 0; l < c->s.L; ++l)
      if (!ok(arrs[i][l]))
        return c->fail(K2_ERR_ARG, "weights.%s[%d] must be a non-null 16-byte aligned device pointer", names[i], l);
  }
  return K2_OK;
}

thread_local std::string g_init_error;

}  // namespace

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// saved cache state (layout documented in include/k2.h)
// ---------------------------------------------------------------------------
namespace {

struct StateHeader {
  char magic[4];
  int32_t version;
  int32_t fp[12];
  int32_t cached, n_tokens;
  int64_t row_bytes, scale_bytes, total_bytes;
  int32_t reserved[2];
};
static_assert(sizeof(StateHeader) == K2_STATE_HEADER_BYTES, "state header size");
static_assert(offsetof(StateHeader, fp) == 8 && offsetof(StateHeader, cached) == 56 &&
                  offsetof(StateHeader, row_bytes) == 64 && offsetof(StateHeader, reserved) == 88,
              "state header layout");
constexpr char kStateMagic[4] = {'K', '2', 'S', 'T'};
constexpr int32_t kStateVersion = 1;

void state_fingerprint(const k2_config& c, int32_t* fp) {
  fp[0] = c.hidden; fp[1] = c.n_layers; fp[2] = c.n_heads; fp[3] = c.n_kv_heads; fp[4] = c.head_dim;
  fp[5] = c.intermediate; fp[6] = c.norm_groups; fp[7] = c.vocab; fp[8] = c.weight_dtype; fp[9] = c.kv_dtype;
  std::memcpy(&fp[10], &c.eps, sizeof(float));
  std::memcpy(&fp[11], &c.rope_theta, sizeof(float));
}

// Byte offsets of a state: tokens right after the header, then per layer
// K rows, V rows and (int8) the K and V scales, each layer 16-byte aligned.
struct StateGeom {
  int64_t row, scale, kv_off, rows_bytes, scales_bytes, per_layer, total;
};
StateGeom state_geom(const k2_config& c, int64_t cached, int64_t n_tokens) {
  StateGeom g;
  g.row = static_cast<int64_t>(c.head_dim) * elt_bytes(c.kv_dtype);
  g.scale = c.kv_dtype == K2_I8 ? 2 : 0;
  g.kv_off = static_cast<int64_t>(align_up(K2_STATE_HEADER_BYTES + 4 * static_cast<size_t>(n_tokens), 16));
  const int64_t rows = static_cast<int64_t>(c.n_kv_heads) * cached;
  g.rows_bytes = rows * g.row;
  g.scales_bytes = rows * g.scale;
  g.per_layer = static_cast<int64_t>(align_up(static_cast<size_t>(2 * g.rows_bytes + 2 * g.scales_bytes), 16));
  g.total = g.kv_off + c.n_layers * g.per_layer;
  return g;
}

// The reason a state cannot be loaded for config c, or null.
const char* state_problem(const k2_config& c, const void* buf, size_t bytes, StateHeader* out) {
  if (!buf || bytes < sizeof(StateHeader)) return "shorter than the state header";
  StateHeader h;
  std::memcpy(&h, buf, sizeof h);
  if (std::memcmp(h.magic, kStateMagic, 4) != 0) return "not a saved k2 cache state (magic)";
  if (h.version != kStateVersion) return "a state version this library does not read";
  int32_t fp[12];
  state_fingerprint(c, fp);
  if (std::memcmp(fp, h.fp, sizeof fp) != 0)
    return "written for another model architecture or KV format (fingerprint differs)";
  if (h.cached < 0 || h.n_tokens < 0 || h.reserved[0] != 0 || h.reserved[1] != 0) return "damaged header";
  const StateGeom g = state_geom(c, h.cached, h.n_tokens);
  if (h.row_bytes != g.row || h.scale_bytes != g.scale || h.total_bytes != g.total) return "damaged header (sizes)";
  if (bytes < static_cast<size_t>(g.total)) return "truncated (shorter than its header says)";
  if (out) *out = h;
  return nullptr;
}

// One K or V (or scale) block of a layer: nkv runs of `run` bytes, cap
// rows apart on the device, back to back in the state.
cudaError_t state_copy(void* dst, const void* src, size_t run, size_t dev_pitch, int nkv, bool to_device,
                       cudaStream_t st) {
  if (run == 0) return cudaSuccess;
  if (to_device)
    return cudaMemcpy2DAsync(dst, dev_pitch, src, run, run, nkv, cudaMemcpyHostToDevice, st);
  return cudaMemcpy2DAsync(dst, run, src, dev_pitch, run, nkv, cudaMemcpyDeviceToHost, st);
}

}  // namespace

extern "C" {

size_t k2_workspace_bytes(const k2_config* cfg) {
  g_init_error = check_config(cfg);
  if (!g_init_error.empty()) return 0;
  return layout_of(*cfg).total;
}

k2_status k2_init_weights(const k2_config* cfg, const k2_weights* w, void* d_workspace, size_t ws_bytes, void* stream,
                          k2_ctx** out) {
  if (!out) return K2_ERR_ARG;
  *out = nullptr;
  const std::string why = check_config(cfg);
  if (!why.empty()) {
    g_init_error = why;
    const bool shape = why.find("multiple") != std::string::npos || why.find("even") != std::string::npos;
    return why.find("not built") != std::string::npos || why.find("not supported") != std::string::npos
               ? K2_ERR_UNSUPPORTED
               : (shape ? K2_ERR_SHAPE : K2_ERR_ARG);
  }
  k2_ctx* c = new k2_ctx();
  c->cfg = *cfg;
  if (cfg->weight_dtype == K2_Q4 || cfg->weight_dtype == K2_F8) c->l2_mask = 0;
  c->s = sizes_of(*cfg);
  c->lay = layout_of(*cfg);
  k2_status st = validate_weights(c, w);
  if (st != K2_OK) {
    g_init_error = c->err;
    delete c;
    return st;
  }
  if (!d_workspace || reinterpret_cast<uintptr_t>(d_workspace) % kAlign) {
    g_init_error = "workspace must be a non-null 256-byte aligned device pointer";
    delete c;
    return K2_ERR_WORKSPACE;
  }
  if (ws_bytes < c->lay.total) {
    char buf[160];
    snprintf(buf, sizeof buf, "workspace too small: %zu bytes given, %zu needed", ws_bytes, c->lay.total);
    g_init_error = buf;
    delete c;
    return K2_ERR_WORKSPACE;
  }
  c->sms = num_sms();
  if (c->sms <= 0) {
    g_init_error = "no CUDA device";
    delete c;
    return K2_ERR_CUDA;
  }
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  c->ws = ws;
  c->seq_len = reinterpret_cast<int*>(ws + c->lay.seq_len);
  c->guard = reinterpret_cast<unsigned*>(ws + c->lay.guard);
  c->am_counter = reinterpret_cast<unsigned*>(ws + c->lay.am_counter);
  c->rope = reinterpret_cast<float2*>(ws + c->lay.rope);
  c->resid = reinterpret_cast<float*>(ws + c->lay.resid);
  c->qkv = reinterpret_cast<float*>(ws + c->lay.qkv);
  c->attn_out = reinterpret_cast<float*>(ws + c->lay.attn_out);
  c->act = reinterpret_cast<float*>(ws + c->lay.act);
  c->am_val = reinterpret_cast<float*>(ws + c->lay.am_val);
  c->am_idx = reinterpret_cast<int*>(ws + c->lay.am_idx);
  c->attn_part = reinterpret_cast<float*>(ws + c->lay.attn_part);
  c->hist = reinterpret_cast<int*>(ws + c->lay.hist);
  c->slog = reinterpret_cast<float*>(ws + c->lay.slog);
  c->embed = w->embed;
  c->lm_head = w->lm_head;
  c->final_norm = w->final_norm;
  for (int l = 0; l < c->s.L; ++l) {
    c->attn_norm.push_back(w->attn_norm[l]);
    c->mlp_norm.push_back(w->mlp_norm[l]);
  }
  c->len.assign(c->s.B, 0);
  if (!plan_all(c)) {
    g_init_error = "no GEMV/attention tiling fits this shape";
    delete c;
    return K2_ERR_UNSUPPORTED;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if ((e = packed_init_attrs()) || (e = attn_init_attrs()) || (e = misc_init_attrs())) {
    g_init_error = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    delete c;
    return K2_ERR_CUDA;
  }
  c->attn_resident = c->sms * attn_ctas_per_sm(c->s.d, c->s.rep, cfg->kv_dtype == K2_F32 ? 0 : cfg->kv_dtype);
  c->attn_cluster_max = attn_max_cluster(c->s.d, c->s.rep, cfg->kv_dtype == K2_F32 ? 0 : cfg->kv_dtype,
                                         kAttnMaxCluster);
  if (c->attn_cluster_max < 1) {
    g_init_error = "no thread-block cluster of the attention kernel fits this GPU";
    delete c;
    return K2_ERR_UNSUPPORTED;
  }
  if (cfg->kv_dtype == K2_F16 && prefill_attn_tc_supported(c->s.d, c->s.rep)) {
    const long long rows = static_cast<long long>(c->s.B) * c->s.nkv * c->lay.cap;
    c->pf_tc = attn_encode_kv_layers(&c->pf_maps.k, c->kc(0), rows, c->s.d, c->s.L, c->lay.kv_layer, 64) &&
               attn_encode_kv_layers(&c->pf_maps.v, c->vc(0), rows, c->s.d, c->s.L, c->lay.kv_layer, 64);
  }
  if (cfg->kv_dtype == K2_F16 && attn_tc_supported(c->s.d, c->s.rep)) {
    c->tm_k.resize(c->s.L);
    c->tm_v.resize(c->s.L);
    const long long rows = static_cast<long long>(c->s.B) * c->s.nkv * c->lay.cap;
    for (int l = 0; l < c->s.L; ++l)
      if (!attn_encode_kv(c->tm_k[l].data(), c->kc(l), rows, c->s.d) ||
          !attn_encode_kv(c->tm_v[l].data(), c->vc(l), rows, c->s.d)) {
        g_init_error = "init: tensor maps of the KV cache";
        delete c;
        return K2_ERR_CUDA;
      }
  }
  // zero the state words (lengths, guard, counters) and build the rope table
  // and the tagged activations (a fresh context must not see an old tag)
  if ((e = cudaMemsetAsync(ws, 0, c->lay.rope, s)) ||
      (e = cudaMemsetAsync(ws + c->lay.t_resid, 0,
                           c->lay.t_part + 8 * static_cast<size_t>(c->s.nkv) * kMegaSplitMax * c->s.rep *
                                               (c->s.d + 2) - c->lay.t_resid,
                           s)) ||
      (e = launch_rope_table(c->rope, c->lay.cap, c->s.d, static_cast<double>(cfg->rope_theta), s))) {
    g_init_error = std::string("init: ") + cudaGetErrorString(e);
    delete c;
    return K2_ERR_CUDA;
  }
  const Sizes& z = c->s;
  if (cfg->weight_dtype == K2_Q4) {  // quantize the bf16 inputs into int4 units (codes + block scales)
    for (int l = 0; l < z.L && e == cudaSuccess; ++l) {
      const auto lay = [](int kind) { return tiled_kind(kind) ? LAYOUT_TILES : LAYOUT_PAIRS; };
      e = launch_q4_pack(static_cast<uint8_t*>(c->wqkv(l)), nullptr, w->wq[l], w->wk[l], w->wv[l], PACK_QKV, z.qkv_n,
                         z.H, z.nq, z.nkv, z.d, lay(0), s);
      if (e == cudaSuccess)
        e = launch_q4_pack(static_cast<uint8_t*>(c->wop(l)), nullptr, w->wo[l], nullptr, nullptr, PACK_PLAIN, z.H,
                           z.nq * z.d, 0, 0, 1, lay(1), s);
      if (e == cudaSuccess)
        e = launch_q4_pack(static_cast<uint8_t*>(c->wgu(l)), nullptr, w->w_gate[l], w->w_up[l], nullptr, PACK_GATEUP,
                           2 * z.I, z.H, 0, 0, 1, lay(2), s);
      if (e == cudaSuccess)
        e = launch_q4_pack(static_cast<uint8_t*>(c->wdown(l)), nullptr, w->w_down[l], nullptr, nullptr, PACK_PLAIN,
                           z.H, z.I, 0, 0, 1, lay(3), s);
    }
    if (e == cudaSuccess)
      e = launch_q4_pack(static_cast<uint8_t*>(c->wlm()), nullptr, w->lm_head, nullptr, nullptr, PACK_PLAIN, z.V, z.H,
                         0, 0, 1, tiled_kind(4) ? LAYOUT_TILES : LAYOUT_PAIRS, s);
  }
  if (cfg->weight_dtype == K2_F8) {  // quantize the bf16 inputs into fp8 rows + scales
    auto sc = [&](size_t base, size_t stride, int l) { return reinterpret_cast<float*>(ws + base + stride * l); };
    const auto lay = [](int kind) { return tiled_kind(kind) ? LAYOUT_TILES : LAYOUT_PAIRS; };
    const auto& L = c->lay;
    for (int l = 0; l < z.L && e == cudaSuccess; ++l) {
      e = launch_quant_pack(static_cast<uint8_t*>(c->wqkv(l)), sc(L.sqkv, L.sqkv_layer, l), w->wq[l], w->wk[l],
                            w->wv[l], PACK_QKV, z.qkv_n, z.H, z.nq, z.nkv, z.d, lay(0), s);
      if (e == cudaSuccess)
        e = launch_quant_pack(static_cast<uint8_t*>(c->wop(l)), sc(L.so, L.so_layer, l), w->wo[l], nullptr, nullptr,
                              PACK_PLAIN, z.H, z.nq * z.d, 0, 0, 1, lay(1), s);
      if (e == cudaSuccess)
        e = launch_quant_pack(static_cast<uint8_t*>(c->wgu(l)), sc(L.sgu, L.sgu_layer, l), w->w_gate[l], w->w_up[l],
                              nullptr, PACK_GATEUP, 2 * z.I, z.H, 0, 0, 1, lay(2), s);
      if (e == cudaSuccess)
        e = launch_quant_pack(static_cast<uint8_t*>(c->wdown(l)), sc(L.sdown, L.sdown_layer, l), w->w_down[l], nullptr,
                              nullptr, PACK_PLAIN, z.H, z.I, 0, 0, 1, lay(3), s);
    }
    if (e == cudaSuccess)
      e = launch_quant_pack(static_cast<uint8_t*>(c->wlm()), reinterpret_cast<float*>(ws + L.slm), w->lm_head, nullptr,
                            nullptr, PACK_PLAIN, z.V, z.H, 0, 0, 1, lay(4), s);
  }
  for (int l = 0; l < z.L && e == cudaSuccess && !quantized(cfg->weight_dtype); ++l) {
    e = launch_pack(c->wqkv(l), w->wq[l], w->wk[l], w->wv[l], PACK_QKV, z.qkv_n, z.H, z.wb, z.nq, z.nkv, z.d, s);
    if (e == cudaSuccess)
      e = launch_pack(c->wop(l), w->wo[l], nullptr, nullptr, PACK_PLAIN, z.H, z.nq * z.d, z.wb, 0, 0, 1, s);
    if (e == cudaSuccess)
      e = launch_pack(c->wgu(l), w->w_gate[l], w->w_up[l], nullptr, PACK_GATEUP, 2 * z.I, z.H, z.wb, 0, 0, 1, s);
    if (e == cudaSuccess)
      e = launch_pack(c->wdown(l), w->w_down[l], nullptr, nullptr, PACK_PLAIN, z.H, z.I, z.wb, 0, 0, 1, s);
  }
  if (e == cudaSuccess && !quantized(cfg->weight_dtype))
    e = launch_pack(c->wlm(), w->lm_head, nullptr, nullptr, PACK_PLAIN, z.V, z.H, z.wb, 0, 0, 1, s);
  for (int l = 0; l < z.L && e == cudaSuccess && cfg->weight_dtype == K2_F8 && c->lay.pchunk > 0; ++l) {
    e = launch_f8_expand(c->tcw(l, 0), static_cast<const uint8_t*>(c->wqkv(l)), z.qkv_n, z.H, tiled_kind(0), s);
    if (e == cudaSuccess)
      e = launch_f8_expand(c->tcw(l, 1), static_cast<const uint8_t*>(c->wop(l)), z.H, z.nq * z.d, tiled_kind(1), s);
    if (e == cudaSuccess)
      e = launch_f8_expand(c->tcw(l, 2), static_cast<const uint8_t*>(c->wgu(l)), 2 * z.I, z.H, tiled_kind(2), s);
    if (e == cudaSuccess)
      e = launch_f8_expand(c->tcw(l, 3), static_cast<const uint8_t*>(c->wdown(l)), z.H, z.I, tiled_kind(3), s);
  }
  if (e != cudaSuccess) {
    g_init_error = std::string("repack: ") + cudaGetErrorString(e);
    delete c;
    return K2_ERR_CUDA;
  }
  if ((e = plan_mega(c, s)) != cudaSuccess) {
    g_init_error = std::string("persistent step set-up: ") + cudaGetErrorString(e);
    delete c;
    return K2_ERR_CUDA;
  }
  if (quantized(cfg->weight_dtype) && !c->mega_ok) {
    g_init_error = "fp8 and int4 weights run on the persistent step only, which this shape / GPU does not support";
    delete c;
    return K2_ERR_UNSUPPORTED;
  }
  if ((e = plan_tc_prefill(c)) != cudaSuccess) {
    g_init_error = std::string("tensor-core prefill set-up: ") + cudaGetErrorString(e);
    delete c;
    return K2_ERR_CUDA;
  }
  *out = c;
  return K2_OK;
}

void k2_free(k2_ctx* c) {
  if (!c) return;
  for (auto& kv : c->graphs) cudaGraphExecDestroy(kv.second);
  for (auto& kv : c->spec_graphs) cudaGraphExecDestroy(kv.second);
  for (cudaEvent_t e : c->pev) cudaEventDestroy(e);
  delete c;
}

const char* k2_last_error(const k2_ctx* c) { return c ? c->err.c_str() : g_init_error.c_str(); }

k2_status k2_get_info(const k2_ctx* c, k2_info* info) {
  if (!c || !info) return K2_ERR_ARG;
  info->kv_capacity = c->lay.cap;
  info->num_sms = c->sms;
  info->attn_splits = attn_splits(c, 1);
  info->gemv_grid = c->grid_gu;
  info->persistent_grid = c->mega_ok ? c->mega_grid : 0;
  info->persistent_splits = c->mega_ok ? c->mega.nsplit : 0;
  info->tc_prefill = c->tc_ok ? 1 : 0;
  info->tc_batched = c->tc_full ? 1 : 0;
  info->kv_bytes = static_cast<int64_t>(c->lay.kv_bytes);
  info->repack_bytes = static_cast<int64_t>(c->lay.repack_bytes);
  info->scratch_bytes = static_cast<int64_t>(c->lay.total - c->lay.kv_bytes - c->lay.repack_bytes);
  return K2_OK;
}

k2_status k2_prefill(k2_ctx* c, int32_t seq, const int32_t* d_tokens, int32_t n, int32_t* d_next_token,
                     float* d_logits, void* stream) {
  if (!c) return K2_ERR_ARG;
  if (seq < 0 || seq >= c->s.B) return c->fail(K2_ERR_ARG, "seq %d outside [0, %d)", seq, c->s.B);
  if (n < 1) return c->fail(K2_ERR_ARG, "n must be >= 1 (got %d)", n);
  if (!d_tokens || !d_next_token) return c->fail(K2_ERR_ARG, "d_tokens and d_next_token must be non-null");
  if (static_cast<long long>(c->len[seq]) + n > c->s.ctx)
    return c->fail(K2_ERR_CONTEXT_FULL, "prompt of %d tokens does not fit: sequence %d holds %d of %d", n, seq,
                   c->len[seq], c->s.ctx);
  float* lg = d_logits ? d_logits : (c->sampling ? c->slog + static_cast<size_t>(seq) * c->s.V : nullptr);
  Launcher ln{c, static_cast<cudaStream_t>(stream), c->pdl};
  if (c->tc_ok && c->use_tc && n >= kTcPrefillMin) {
    const cudaError_t e = prefill_tc(c, seq, d_tokens, n, d_next_token, lg, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return c->cuda_fail(e, "tensor-core prefill");
  } else {
    for (int i = 0; i < n; ++i) {
      const bool last = i == n - 1;
      enqueue_token(c, ln, seq, d_tokens + i, nullptr, d_next_token, last ? lg : nullptr, last);
    }
  }
  if (c->sampling) {
    ln.pdl = false;
    enqueue_sample(c, ln, lg, 1, c->hist + static_cast<size_t>(seq) * c->lay.cap, c->lay.cap, c->seq_len + seq,
                   c->seq_len + seq, seq, d_next_token);
  }
  if (ln.err != cudaSuccess) return c->cuda_fail(ln.err, "prefill launch");
  c->len[seq] += n;
  return K2_OK;
}

k2_status k2_decode_step(k2_ctx* c, const int32_t* d_tokens, int32_t batch, int32_t* d_next, float* d_logits,
                         void* stream) {
  if (!c) return K2_ERR_ARG;
  if (batch < 1 || batch > c->s.B) return c->fail(K2_ERR_ARG, "batch %d outside [1, %d]", batch, c->s.B);
  if (!d_tokens || !d_next) return c->fail(K2_ERR_ARG, "d_tokens and d_next must be non-null");
  for (int b = 0; b < batch; ++b)
    if (c->len[b] >= c->s.ctx)
      return c->fail(K2_ERR_CONTEXT_FULL, "sequence %d is at max_context %d", b, c->s.ctx);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c->graph) {
    if (!s) return c->fail(K2_ERR_ARG, "graph mode needs a non-default stream");
    auto key = std::make_tuple(batch, static_cast<const void*>(d_tokens), static_cast<const void*>(d_next),
                               static_cast<const void*>(d_logits), stream);
    auto it = c->graphs.find(key);
    if (it == c->graphs.end()) {
      cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
      if (e) return c->cuda_fail(e, "cudaStreamBeginCapture");
      Launcher ln{c, s, c->pdl};
      enqueue_decode(c, ln, d_tokens, batch, d_next, d_logits);
      cudaGraph_t g = nullptr;
      e = cudaStreamEndCapture(s, &g);
      if (ln.err) {
        if (g) cudaGraphDestroy(g);
        return c->cuda_fail(ln.err, "decode capture");
      }
      if (e) return c->cuda_fail(e, "cudaStreamEndCapture");
      cudaGraphExec_t ge = nullptr;
      e = cudaGraphInstantiate(&ge, g, 0);
      cudaGraphDestroy(g);
      if (e) return c->cuda_fail(e, "cudaGraphInstantiate");
      it = c->graphs.emplace(key, ge).first;
    }
    cudaError_t e = cudaGraphLaunch(it->second, s);
    if (e) return c->cuda_fail(e, "cudaGraphLaunch");
  } else {
    Launcher ln{c, s, c->pdl};
    enqueue_decode(c, ln, d_tokens, batch, d_next, d_logits);
    if (ln.err) return c->cuda_fail(ln.err, "decode launch");
  }
  for (int b = 0; b < batch; ++b) c->len[b] += 1;
  return K2_OK;
}

k2_status k2_decode_layers(k2_ctx* c, float* d_x, int32_t batch, void* stream) {
  if (!c) return K2_ERR_ARG;
  if (batch < 1 || batch > c->s.B) return c->fail(K2_ERR_ARG, "batch %d outside [1, %d]", batch, c->s.B);
  if (!d_x || reinterpret_cast<uintptr_t>(d_x) % 16) return c->fail(K2_ERR_ARG, "d_x must be 16-byte aligned");
  for (int b = 0; b < batch; ++b)
    if (c->len[b] >= c->s.ctx)
      return c->fail(K2_ERR_CONTEXT_FULL, "sequence %d is at max_context %d", b, c->s.ctx);
  Launcher ln{c, static_cast<cudaStream_t>(stream), c->pdl};
  for (int b = 0; b < batch; ++b)
    enqueue_token(c, ln, b, nullptr, d_x + static_cast<size_t>(b) * c->s.H, nullptr, nullptr, false);
  if (ln.err) return c->cuda_fail(ln.err, "layers launch");
  for (int b = 0; b < batch; ++b) c->len[b] += 1;
  return K2_OK;
}

k2_status k2_kv_reset(k2_ctx* c, int32_t seq, void* stream) {
  if (!c) return K2_ERR_ARG;
  if (seq < -1 || seq >= c->s.B) return c->fail(K2_ERR_ARG, "seq %d outside [-1, %d)", seq, c->s.B);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (seq == -1) {
    e = cudaMemsetAsync(c->seq_len, 0, sizeof(int) * c->s.B, s);
    if (e) return c->cuda_fail(e, "kv_reset");
    c->len.assign(c->s.B, 0);
  } else {
    e = cudaMemsetAsync(c->seq_len + seq, 0, sizeof(int), s);
    if (e) return c->cuda_fail(e, "kv_reset");
    c->len[seq] = 0;
  }
  return K2_OK;
}

k2_status k2_kv_set_len(k2_ctx* c, int32_t seq, int32_t len, void* stream) {
  if (!c) return K2_ERR_ARG;
  if (seq < 0 || seq >= c->s.B) return c->fail(K2_ERR_ARG, "seq %d outside [0, %d)", seq, c->s.B);
  if (len < 0 || len > c->s.ctx) return c->fail(K2_ERR_CONTEXT_FULL, "len %d outside [0, %d]", len, c->s.ctx);
  // a kernel-free host->device write of one int: pageable copies are staged
  // synchronously by the driver, so the source may go out of scope
  static thread_local int v;
  v = len;
  cudaError_t e = cudaMemcpyAsync(c->seq_len + seq, &v, sizeof(int), cudaMemcpyHostToDevice,
                                  static_cast<cudaStream_t>(stream));
  if (e) return c->cuda_fail(e, "kv_set_len");
  e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e) return c->cuda_fail(e, "kv_set_len");
  c->len[seq] = len;
  return K2_OK;
}

k2_status k2_kv_view(k2_ctx* c, int32_t layer, int32_t seq, void** k, void** v, void** k_scale, void** v_scale,
                     int32_t* len) {
  if (!c) return K2_ERR_ARG;
  if (layer < 0 || layer >= c->s.L || seq < 0 || seq >= c->s.B)
    return c->fail(K2_ERR_ARG, "layer %d / seq %d out of range", layer, seq);
  const size_t per_seq = static_cast<size_t>(c->s.nkv) * c->lay.cap;
  const size_t off = static_cast<size_t>(seq) * per_seq;
  if (k) *k = static_cast<uint8_t*>(c->kc(layer)) + off * c->s.d * c->s.kvb;
  if (v) *v = static_cast<uint8_t*>(c->vc(layer)) + off * c->s.d * c->s.kvb;
  if (k_scale) *k_scale = c->ks(layer) ? static_cast<uint8_t*>(c->ks(layer)) + off * 2 : nullptr;
  if (v_scale) *v_scale = c->vs(layer) ? static_cast<uint8_t*>(c->vs(layer)) + off * 2 : nullptr;
  if (len) *len = c->len[seq];
  return K2_OK;
}

k2_status k2_hidden_view(k2_ctx* c, int32_t b, float** d_x) {
  if (!c || !d_x) return K2_ERR_ARG;
  if (b < 0 || b >= c->s.B) return c->fail(K2_ERR_ARG, "slot %d out of range", b);
  *d_x = c->resid + static_cast<size_t>(b) * c->s.H;
  return K2_OK;
}

k2_status k2_spec_logits_view(k2_ctx* c, float** d_logits, int32_t* rows) {
  if (!c || !d_logits || !rows) return K2_ERR_ARG;
  *d_logits = c->lay.pchunk > 0 ? reinterpret_cast<float*>(c->ws + c->lay.vlog) : nullptr;
  *rows = c->spec_rows;
  return K2_OK;
}

k2_status k2_sync_status(k2_ctx* c, void* stream) {
  if (!c) return K2_ERR_ARG;
  unsigned g = 0;
  cudaError_t e = cudaMemcpyAsync(&g, c->guard, sizeof g, cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream));
  if (!e) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e) return c->cuda_fail(e, "sync_status");
  if (g == 0) return K2_OK;
  std::string why;
  if (g & GUARD_TOKEN) why += " token-id-out-of-range";
  if (g & GUARD_TIMEOUT) why += " bounded-wait-timeout";
  if (g & GUARD_NAN) why += " nan-logit";
  if (g & GUARD_POS) why += " position-outside-cache";
  if (g & GUARD_RANGE) why += " beyond-fp16-range";
  return c->fail(K2_ERR_DEVICE_GUARD, "device guard 0x%x:%s", g, why.c_str());
}

k2_status k2_clear_status(k2_ctx* c, void* stream) {
  if (!c) return K2_ERR_ARG;
  cudaError_t e = cudaMemsetAsync(c->guard, 0, sizeof(unsigned), static_cast<cudaStream_t>(stream));
  // a step cut short by a timeout may have left the grid barrier half counted
  // the finished-CTA counter (not the epoch: tags must stay fresh)
  if (!e) e = cudaMemsetAsync(c->ws + c->lay.msync, 0, sizeof(unsigned), static_cast<cudaStream_t>(stream));
  // a step that failed on the device left its sequences' lengths where they
  // were, while the host copy advanced when the step was enqueued: take the
  // device's word for it
  std::vector<int> dlen(c->s.B, 0);
  if (!e)
    e = cudaMemcpyAsync(dlen.data(), c->seq_len, sizeof(int) * c->s.B, cudaMemcpyDeviceToHost,
                        static_cast<cudaStream_t>(stream));
  if (!e) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e) return c->cuda_fail(e, "clear_status");
  for (int b = 0; b < c->s.B; ++b) c->len[b] = dlen[b];
  return K2_OK;
}

k2_status k2_set_option(k2_ctx* c, int32_t option, int64_t value) {
  if (!c) return K2_ERR_ARG;
  switch (option) {
    case K2_OPT_PDL: c->pdl = value != 0; break;
    case K2_OPT_GRAPH: c->graph = value != 0; break;
    case K2_OPT_PERSISTENT:
      if (value == 0 && quantized(c->cfg.weight_dtype))
        return c->fail(K2_ERR_UNSUPPORTED, "fp8 and int4 weights run on the persistent step only");
      c->use_mega = value != 0;
      break;
    case K2_OPT_TC_PREFILL: c->use_tc = value != 0; break;
    case K2_OPT_TC_DECODE: c->use_tc_decode = value != 0; break;
    case K2_OPT_ATTN_SPLITS:
      if (value < 0 || value > kAttnMaxCluster)
        return c->fail(K2_ERR_ARG, "splits %lld outside [0, %d]", (long long)value, kAttnMaxCluster);
      c->force_splits = static_cast<int>(value);
      break;
    case K2_OPT_WAIT_LIMIT_US:
      if (value < 1 || value > 1000000)
        return c->fail(K2_ERR_ARG, "wait limit %lld us outside [1, 1000000]", (long long)value);
      c->poll_limit_ns = static_cast<unsigned long long>(value) * 1000ull;
      break;
    case K2_OPT_L2_AHEAD:
      if (value < 0 || value > 64) return c->fail(K2_ERR_ARG, "L2 look-ahead %lld outside [0, 64]", (long long)value);
      c->l2_ahead = static_cast<int>(value);
      break;
    case K2_OPT_L2_AHEAD_PHASES:
      if (value < 0 || value > 63) return c->fail(K2_ERR_ARG, "phase mask %lld outside [0, 63]", (long long)value);
      c->l2_mask = static_cast<int>(value);
      break;
    case K2_OPT_PREFILL_ATTN: c->use_pf_tc = value != 0; break;
    case K2_OPT_PREFILL_GEMM: c->pf_whole = value != 0; break;
    case K2_OPT_PREFILL_SPLIT:
      if (value < 0 || value > 3) return c->fail(K2_ERR_ARG, "prefill split %lld outside [0, 3]", (long long)value);
      c->pf_split = static_cast<int>(value);
      break;
    case K2_OPT_TRACE:
      if (value < 0 || value % 8) return c->fail(K2_ERR_ARG, "trace buffer must be 8-byte aligned (or 0)");
      c->trace = reinterpret_cast<unsigned long long*>(static_cast<uintptr_t>(value));
      break;
    case K2_OPT_STALL_PHASE:
      if (value < -1 || value == 0 || value > 5LL * c->s.L)
        return c->fail(K2_ERR_ARG, "stall phase %lld outside -1 or [1, %d]", (long long)value, 5 * c->s.L);
      c->stall_phase = static_cast<int>(value);
      break;
    default: return c->fail(K2_ERR_ARG, "unknown option %d", option);
  }
  for (auto& kv : c->graphs) cudaGraphExecDestroy(kv.second);
  for (auto& kv : c->spec_graphs) cudaGraphExecDestroy(kv.second);
  c->graphs.clear();
  c->spec_graphs.clear();
  return K2_OK;
}

k2_status k2_profile_decode(k2_ctx* c, const int32_t* d_tokens, int32_t batch, int32_t* d_next, float* ms,
                            int32_t* launches, void* stream) {
  if (!c || !ms || !launches) return K2_ERR_ARG;
  if (batch < 1 || batch > c->s.B) return c->fail(K2_ERR_ARG, "batch %d outside [1, %d]", batch, c->s.B);
  if (!d_tokens || !d_next) return c->fail(K2_ERR_ARG, "d_tokens and d_next must be non-null");
  for (int b = 0; b < batch; ++b)
    if (c->len[b] >= c->s.ctx)
      return c->fail(K2_ERR_CONTEXT_FULL, "sequence %d is at max_context %d", b, c->s.ctx);
  Launcher ln{c, static_cast<cudaStream_t>(stream), false};
  ln.profile = true;
  enqueue_decode(c, ln, d_tokens, batch, d_next, nullptr);
  if (ln.collect(ms, launches) != cudaSuccess) return c->cuda_fail(ln.err, "profile launch");
  for (int b = 0; b < batch; ++b) c->len[b] += 1;
  return K2_OK;
}


k2_status k2_kv_state_bytes(const k2_ctx* c, int32_t seq, int32_t n_tokens, size_t* bytes) {
  if (!c || !bytes || seq < 0 || seq >= c->s.B || n_tokens < 0) return K2_ERR_ARG;
  *bytes = static_cast<size_t>(state_geom(c->cfg, c->len[seq], n_tokens).total);
  return K2_OK;
}

k2_status k2_kv_save(k2_ctx* c, int32_t seq, const int32_t* h_tokens, int32_t n_tokens, void* h_buf,
                     size_t buf_bytes, size_t* written, void* stream) {
  if (!c) return K2_ERR_ARG;
  if (seq < 0 || seq >= c->s.B) return c->fail(K2_ERR_ARG, "seq %d outside [0, %d)", seq, c->s.B);
  if (n_tokens < 0 || (n_tokens > 0 && !h_tokens) || !h_buf)
    return c->fail(K2_ERR_ARG, "h_buf and (for n_tokens > 0) h_tokens must be non-null");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int cached = c->len[seq];
  const StateGeom g = state_geom(c->cfg, cached, n_tokens);
  if (buf_bytes < static_cast<size_t>(g.total))
    return c->fail(K2_ERR_WORKSPACE, "the state needs %lld bytes, the buffer has %zu", (long long)g.total, buf_bytes);
  // the cache must hold what the host believes: no pending fault, same length
  unsigned guard = 0;
  int dev_len = -1;
  cudaError_t e = cudaMemcpyAsync(&guard, c->guard, sizeof guard, cudaMemcpyDeviceToHost, st);
  if (!e) e = cudaMemcpyAsync(&dev_len, c->seq_len + seq, sizeof dev_len, cudaMemcpyDeviceToHost, st);
  if (!e) e = cudaStreamSynchronize(st);
  if (e) return c->cuda_fail(e, "kv_save");
  if (guard) return c->fail(K2_ERR_DEVICE_GUARD, "the device guard is set (0x%x): not saving", guard);
  if (dev_len != cached)
    return c->fail(K2_ERR_DEVICE_GUARD, "sequence %d holds %d rows on the device, %d on the host", seq, dev_len, cached);
  uint8_t* out = static_cast<uint8_t*>(h_buf);
  StateHeader h = {};
  std::memcpy(h.magic, kStateMagic, 4);
  h.version = kStateVersion;
  state_fingerprint(c->cfg, h.fp);
  h.cached = cached;
  h.n_tokens = n_tokens;
  h.row_bytes = g.row;
  h.scale_bytes = g.scale;
  h.total_bytes = g.total;
  std::memcpy(out, &h, sizeof h);
  if (n_tokens) std::memcpy(out + sizeof h, h_tokens, 4 * static_cast<size_t>(n_tokens));
  std::memset(out + sizeof h + 4 * static_cast<size_t>(n_tokens), 0,
              static_cast<size_t>(g.kv_off) - sizeof h - 4 * static_cast<size_t>(n_tokens));
  const size_t head0 = static_cast<size_t>(seq) * c->s.nkv * c->lay.cap;  // row of (seq, head 0)
  const size_t run = static_cast<size_t>(cached) * g.row, srun = static_cast<size_t>(cached) * g.scale;
  for (int l = 0; l < c->s.L && !e; ++l) {
    uint8_t* o = out + g.kv_off + static_cast<size_t>(l) * g.per_layer;
    const size_t pitch = static_cast<size_t>(c->lay.cap) * g.row;
    e = state_copy(o, static_cast<uint8_t*>(c->kc(l)) + head0 * g.row, run, pitch, c->s.nkv, false, st);
    if (!e) e = state_copy(o + g.rows_bytes, static_cast<uint8_t*>(c->vc(l)) + head0 * g.row, run, pitch, c->s.nkv, false, st);
    if (!e && g.scale) {
      const size_t sp = static_cast<size_t>(c->lay.cap) * 2;
      e = state_copy(o + 2 * g.rows_bytes, static_cast<uint8_t*>(c->ks(l)) + head0 * 2, srun, sp, c->s.nkv, false, st);
      if (!e)
        e = state_copy(o + 2 * g.rows_bytes + g.scales_bytes, static_cast<uint8_t*>(c->vs(l)) + head0 * 2, srun, sp,
                       c->s.nkv, false, st);
    }
    const size_t used = static_cast<size_t>(2 * g.rows_bytes + 2 * g.scales_bytes);
    std::memset(o + used, 0, static_cast<size_t>(g.per_layer) - used);
  }
  if (!e) e = cudaStreamSynchronize(st);
  if (e) return c->cuda_fail(e, "kv_save copies");
  if (written) *written = static_cast<size_t>(g.total);
  return K2_OK;
}

k2_status k2_kv_peek(const k2_config* cfg, const void* h_buf, size_t buf_bytes, int32_t* cached, int32_t* n_tokens) {
  if (!cfg) return K2_ERR_ARG;
  StateHeader h;
  if (state_problem(*cfg, h_buf, buf_bytes, &h)) return K2_ERR_STATE;
  if (cached) *cached = h.cached;
  if (n_tokens) *n_tokens = h.n_tokens;
  return K2_OK;
}

k2_status k2_kv_load(k2_ctx* c, int32_t seq, const void* h_buf, size_t buf_bytes, int32_t* h_tokens,
                     int32_t max_tokens, void* stream) {
  if (!c) return K2_ERR_ARG;
  if (seq < 0 || seq >= c->s.B) return c->fail(K2_ERR_ARG, "seq %d outside [0, %d)", seq, c->s.B);
  StateHeader h;
  if (const char* why = state_problem(c->cfg, h_buf, buf_bytes, &h)) return c->fail(K2_ERR_STATE, "refusing the state: %s", why);
  if (h.cached > c->s.ctx)
    return c->fail(K2_ERR_CONTEXT_FULL, "the state holds %d rows, this context's max_context is %d", h.cached, c->s.ctx);
  if (h.n_tokens > max_tokens || (h.n_tokens > 0 && !h_tokens))
    return c->fail(K2_ERR_ARG, "the state holds %d token ids, h_tokens has room for %d", h.n_tokens,
                   h_tokens ? max_tokens : 0);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const StateGeom g = state_geom(c->cfg, h.cached, h.n_tokens);
  const uint8_t* in = static_cast<const uint8_t*>(h_buf);
  const size_t head0 = static_cast<size_t>(seq) * c->s.nkv * c->lay.cap;
  const size_t run = static_cast<size_t>(h.cached) * g.row, srun = static_cast<size_t>(h.cached) * g.scale;
  cudaError_t e = cudaSuccess;
  for (int l = 0; l < c->s.L && !e; ++l) {
    const uint8_t* o = in + g.kv_off + static_cast<size_t>(l) * g.per_layer;
    const size_t pitch = static_cast<size_t>(c->lay.cap) * g.row;
    e = state_copy(static_cast<uint8_t*>(c->kc(l)) + head0 * g.row, o, run, pitch, c->s.nkv, true, st);
    if (!e) e = state_copy(static_cast<uint8_t*>(c->vc(l)) + head0 * g.row, o + g.rows_bytes, run, pitch, c->s.nkv, true, st);
    if (!e && g.scale) {
      const size_t sp = static_cast<size_t>(c->lay.cap) * 2;
      e = state_copy(static_cast<uint8_t*>(c->ks(l)) + head0 * 2, o + 2 * g.rows_bytes, srun, sp, c->s.nkv, true, st);
      if (!e)
        e = state_copy(static_cast<uint8_t*>(c->vs(l)) + head0 * 2, o + 2 * g.rows_bytes + g.scales_bytes, srun, sp,
                       c->s.nkv, true, st);
    }
  }
  // the saved ids of the cached rows become the sequence's token history
  const int nh = std::min(h.cached, h.n_tokens);
  if (!e && nh > 0)
    e = cudaMemcpyAsync(c->hist + static_cast<size_t>(seq) * c->lay.cap, in + sizeof(StateHeader),
                        sizeof(int) * static_cast<size_t>(nh), cudaMemcpyHostToDevice, st);
  // the length goes last, from a buffer that outlives the copy (synchronised below)
  static thread_local int v;
  v = h.cached;
  if (!e) e = cudaMemcpyAsync(c->seq_len + seq, &v, sizeof(int), cudaMemcpyHostToDevice, st);
  if (!e) e = cudaStreamSynchronize(st);
  if (e) return c->cuda_fail(e, "kv_load copies");
  c->len[seq] = h.cached;
  if (h.n_tokens) std::memcpy(h_tokens, in + sizeof(StateHeader), 4 * static_cast<size_t>(h.n_tokens));
  return K2_OK;
}


k2_status k2_set_sampling(k2_ctx* c, const k2_sampling* p) {
  if (!c) return K2_ERR_ARG;
  if (p) {
    if (!(p->temperature >= 0.f) || !(p->top_p > 0.f && p->top_p <= 1.f) || !(p->min_p >= 0.f && p->min_p <= 1.f) ||
        !(p->repetition_penalty > 0.f) || p->top_k < 0 || !std::isfinite(p->temperature) ||
        !std::isfinite(p->repetition_penalty))
      return c->fail(K2_ERR_ARG,
                     "sampling needs temperature >= 0, top_k >= 0, top_p in (0, 1], min_p in [0, 1], "
                     "repetition_penalty > 0 (all finite)");
  }
  const bool on = p && p->temperature > 0.f;
  if (on && c->sample_cpr.empty()) {
    c->sample_cpr.assign(c->s.B + 1, 0);
    for (int r = 1; r <= c->s.B; ++r) {
      c->sample_cpr[r] = sample_ctas_per_row(r, c->s.V);
      if (c->sample_cpr[r] < 1) {
        c->sample_cpr.clear();
        return c->fail(K2_ERR_UNSUPPORTED, "the sampler cannot hold %d rows of a %d-token vocabulary", r, c->s.V);
      }
    }
  }
  c->samp = on ? *p : k2_sampling{};
  c->sampling = on;
  for (auto& kv : c->graphs) cudaGraphExecDestroy(kv.second);
  for (auto& kv : c->spec_graphs) cudaGraphExecDestroy(kv.second);
  c->graphs.clear();
  c->spec_graphs.clear();
  return K2_OK;
}

k2_status k2_sample_logits(k2_ctx* c, const float* d_logits, int32_t rows, const int32_t* d_seen,
                           int32_t seen_stride, const int32_t* d_seen_len, const int32_t* d_position,
                           int32_t first_seq, int32_t* d_next, void* stream) {
  if (!c) return K2_ERR_ARG;
  if (!c->sampling) return c->fail(K2_ERR_ARG, "sampling is not set (temperature 0)");
  if (rows < 1 || rows > c->s.B) return c->fail(K2_ERR_ARG, "rows %d outside [1, %d]", rows, c->s.B);
  if (!d_logits || !d_position || !d_next || (d_seen && (!d_seen_len || seen_stride < 0)))
    return c->fail(K2_ERR_ARG, "d_logits, d_position, d_next (and d_seen_len with d_seen) must be non-null");
  Launcher ln{c, static_cast<cudaStream_t>(stream), false};
  enqueue_sample(c, ln, d_logits, rows, d_seen, seen_stride, d_seen_len, d_position, first_seq, d_next);
  if (ln.err != cudaSuccess) return c->cuda_fail(ln.err, "sample launch");
  return K2_OK;
}

k2_status k2_philox(uint32_t first, int32_t n, uint32_t c1, uint32_t c2, uint32_t c3, uint64_t key, uint32_t* d_out,
                    void* stream) {
  if (n < 0 || (n > 0 && !d_out)) return K2_ERR_ARG;
  const cudaError_t e = launch_philox(first, n, c1, c2, c3, static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32),
                                      d_out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? K2_OK : K2_ERR_CUDA;
}

// Drafting works on the history read backwards, r[k] = h_tokens[T - 1 - k].
// The Z-algorithm gives, for every shift i >= 1, z[i] = the length of the
// longest common prefix of r and r[i..]: the number of ids that the earlier
// stretch of the history ending at position T - 1 - i shares with the end of
// the history.  A suffix of n ids occurred earlier, ending at T - 1 - i,
// exactly when z[i] >= n, and the smallest such shifts are its most recent
// occurrences; one pass serves n = 4 and n = 3 alike.
int32_t k2_spec_draft(const int32_t* h_tokens, int32_t n_tokens, int32_t max_draft, int32_t* h_out) {
  if (!h_tokens || n_tokens < 0 || max_draft < 1 || !h_out) return 0;
  constexpr int kLongest = 4, kShortest = 3;
  const int T = n_tokens;
  if (T < kShortest + 1) return 0;
  const int cap = std::min<int>(max_draft, kSpecMax);
  auto r = [&](int k) { return h_tokens[T - 1 - k]; };
  static thread_local std::vector<int> z;
  z.assign(T, 0);
  // shifts of the two most recent occurrences per suffix length n (0 = none)
  int near[kLongest + 1][2] = {};
  for (int i = 1, lo = 0, hi = 0; i + kShortest <= T; ++i) {
    int m = i < hi ? std::min(hi - i, z[i - lo]) : 0;
    while (i + m < T && r(m) == r(i + m)) ++m;
    z[i] = m;
    if (i + m > hi) lo = i, hi = i + m;
    for (int n = kShortest; n <= std::min(m, kLongest); ++n)
      if (i + n <= T) {
        if (!near[n][0]) near[n][0] = i;
        else if (!near[n][1]) near[n][1] = i;
      }
    if (near[kLongest][1]) break;  // both lengths have their two latest occurrences
  }
  for (int n = kLongest; n >= kShortest; --n) {
    const int a = near[n][0], b = near[n][1];
    if (!a) continue;
    // the ids after the newest occurrence run from T - a to the end (a of them)
    int len = std::min(cap, a);
    if (b) {
      // the older occurrence must agree, and its continuation (from T - b)
      // must stay short of the newest occurrence, which starts at T - a - n
      len = std::min(len, b - a - n);
      int agree = 0;
      while (agree < len && h_tokens[T - a + agree] == h_tokens[T - b + agree]) ++agree;
      len = agree;
    }
    if (len > 0) {
      std::copy(h_tokens + T - a, h_tokens + T - a + len, h_out);
      return len;
    }
  }
  return 0;
}

k2_status k2_decode_speculative(k2_ctx* c, int32_t seq, const int32_t* h_tokens, int32_t n_tokens,
                                int32_t max_draft, int32_t* h_out, int32_t* n_out, void* stream) {
  if (!c) return K2_ERR_ARG;
  if (seq < 0 || seq >= c->s.B) return c->fail(K2_ERR_ARG, "seq %d outside [0, %d)", seq, c->s.B);
  if (!h_tokens || !h_out || !n_out || max_draft < 0)
    return c->fail(K2_ERR_ARG, "h_tokens, h_out and n_out must be non-null, max_draft >= 0");
  if (n_tokens != c->len[seq] + 1)
    return c->fail(K2_ERR_ARG, "h_tokens must hold the %d cached ids and the next input (got %d ids)", c->len[seq],
                   n_tokens);
  if (c->sampling) return c->fail(K2_ERR_UNSUPPORTED, "speculative decoding verifies greedy ids only");
  if (c->len[seq] >= c->s.ctx) return c->fail(K2_ERR_CONTEXT_FULL, "sequence %d is at max_context %d", seq, c->s.ctx);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int ids[kSpecMax + 1];
  ids[0] = h_tokens[n_tokens - 1];
  int nd = c->tc_full ? k2_spec_draft(h_tokens, n_tokens, std::min<int>(max_draft, kSpecMax), ids + 1) : 0;
  nd = std::min(nd, c->s.ctx - c->len[seq] - 1);  // every verified row must fit
  if (nd < 0) nd = 0;
  int* d_ids = reinterpret_cast<int*>(c->ws + c->lay.vids);
  int* d_arg = reinterpret_cast<int*>(c->ws + c->lay.varg);
  static thread_local int h_ids[kSpecMax + 1];
  std::copy(ids, ids + nd + 1, h_ids);
  cudaError_t e = cudaMemcpyAsync(d_ids, h_ids, sizeof(int) * (nd + 1), cudaMemcpyHostToDevice, st);
  int out[kSpecMax + 1];
  int accepted = 0;
  // The step's launches read every position on the device, so with
  // K2_OPT_GRAPH they are recorded once per (sequence, block size) and replayed.
  auto run = [&](int nblk, auto&& enqueue) -> cudaError_t {
    if (!c->graph || !st) return enqueue();
    const auto key = std::make_tuple(seq, nblk, stream);
    auto it = c->spec_graphs.find(key);
    if (it == c->spec_graphs.end()) {
      cudaError_t ce = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
      if (ce) return ce;
      const cudaError_t le = enqueue();
      cudaGraph_t g = nullptr;
      ce = cudaStreamEndCapture(st, &g);
      if (le || ce) {
        if (g) cudaGraphDestroy(g);
        return le ? le : ce;
      }
      cudaGraphExec_t ge = nullptr;
      ce = cudaGraphInstantiate(&ge, g, 0);
      cudaGraphDestroy(g);
      if (ce) return ce;
      it = c->spec_graphs.emplace(key, ge).first;
    }
    return cudaGraphLaunch(it->second, st);
  };
  // the logits of every verified position stay in the verification buffer
  // (k2_spec_logits_view); a plain step leaves its one row there too
  float* vlog = c->lay.pchunk > 0 ? reinterpret_cast<float*>(c->ws + c->lay.vlog) : nullptr;
  c->spec_rows = 0;
  if (nd == 0) {  // no draft: an ordinary decode step of this sequence
    if (!e)
      e = run(0, [&] {
        Launcher ln{c, st, false};
        enqueue_token(c, ln, seq, d_ids, nullptr, d_arg, vlog, true);
        return ln.err;
      });
    if (!e) e = cudaMemcpyAsync(out, d_arg, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (!e) e = cudaStreamSynchronize(st);
    if (e) return c->cuda_fail(e, "speculative step");
    c->len[seq] += 1;
    c->spec_rows = vlog ? 1 : 0;
  } else {
    if (!e) e = run(nd + 1, [&] { return verify_block(c, seq, d_ids, nd + 1, d_arg, st); });
    if (!e) e = cudaMemcpyAsync(out, d_arg, sizeof(int) * (nd + 1), cudaMemcpyDeviceToHost, st);
    if (!e) e = cudaStreamSynchronize(st);
    if (e) return c->cuda_fail(e, "speculative verification");
    // draft i is kept while it is the greedy id after the ids before it
    while (accepted < nd && ids[1 + accepted] == out[accepted]) ++accepted;
    const int len = c->len[seq] + 1 + accepted;  // the input row and the accepted drafts
    static thread_local int v;
    v = len;
    e = cudaMemcpyAsync(c->seq_len + seq, &v, sizeof(int), cudaMemcpyHostToDevice, st);
    if (!e) e = cudaStreamSynchronize(st);
    if (e) return c->cuda_fail(e, "speculative length");
    c->len[seq] = len;
    c->spec_rows = nd + 1;
  }
  std::copy(out, out + accepted + 1, h_out);
  *n_out = accepted + 1;
  return K2_OK;
}

k2_status k2_quantize_fp8(const void* d_src, int32_t rows, int32_t cols, uint8_t* d_codes, float* d_scales,
                          void* stream) {
  if (!d_src || !d_codes || !d_scales || rows < 0 || cols < 1) return K2_ERR_ARG;
  const cudaError_t e = launch_quant_pack(d_codes, d_scales, d_src, nullptr, nullptr, PACK_PLAIN, rows, cols, 0, 0, 1,
                                          LAYOUT_PLAIN, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? K2_OK : K2_ERR_CUDA;
}

k2_status k2_quantize_q4(const void* d_src, int32_t rows, int32_t cols, int8_t* d_codes, float* d_scales,
                         void* stream) {
  if (!d_src || !d_codes || !d_scales || rows < 0 || cols < 1) return K2_ERR_ARG;
  const cudaError_t e = launch_q4_pack(reinterpret_cast<uint8_t*>(d_codes), d_scales, d_src, nullptr, nullptr,
                                       PACK_PLAIN, rows, cols, 0, 0, 1, LAYOUT_PLAIN, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? K2_OK : K2_ERR_CUDA;
}
}  // extern "C"
