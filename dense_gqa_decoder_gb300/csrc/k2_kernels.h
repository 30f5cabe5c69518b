// Argument blocks and launchers of the sm_103a kernels (internal to libk2).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace k2 {

// bits of the device guard word (read back by k2_sync_status)
enum : uint32_t {
  GUARD_TOKEN = 1u,    // a token id outside [0, vocab)
  GUARD_TIMEOUT = 2u,  // a bounded wait ran out
  GUARD_NAN = 4u,      // a NaN logit
  GUARD_POS = 8u,      // a position outside the cache
  GUARD_RANGE = 16u,   // a weight or activation outside the fp16 range (fp16 prefill operands)
};

// ---------------------------------------------------------------------------
// streaming GEMV: y = W . norm(x), W [N, K] row-major, one fp32 vector x
// ---------------------------------------------------------------------------
enum GemvEpi : int {
  EPI_STORE = 0,   // out[row] = y
  EPI_RESID = 1,   // out[row] += y   (residual add, in place)
  EPI_QKV = 2,     // row pairs (i, i + d/2) of a head -> split-half RoPE -> out
  EPI_SWIGLU = 3,  // row pairs (gate_i, up_i) -> out[i] = silu(gate) * up
  EPI_ARGMAX = 4,  // logits (optional store) + first-index argmax -> token
};

struct GemvArgs {
  const void* W;
  int N, K;
  const float* x;       // [K]
  const void* gain;     // [K] norm gain in the weight dtype, or null (no norm)
  int groups;
  float eps;
  // tiling (host-chosen)
  int R;       // rows per stage
  int nslice;  // K slices; R * nslice == 8 warps
  int kc;      // 16-byte chunks per lane per slice (<= kGemvKcMax)
  int align;   // CTA row ranges are multiples of this (2 for pair epilogues)
  int nstage;  // ring depth
  uint32_t stage_bytes;
  // epilogue
  float* out;
  const float2* rope;  // [cap][d/2] (cos, sin)
  int cap;             // rows of the rope table (positions 0 .. cap-1)
  int* seq_len;        // position of the token = seq_len[seq] (advanced by EPI_ARGMAX)
  int seq;
  int head_dim;
  int n_rot_heads;  // heads [0, n_rot_heads) are rotated (q and k), the rest (v) are not
  // argmax
  float* logits;      // nullable
  float* part_val;    // [gridDim]
  int* part_idx;      // [gridDim]
  unsigned* counter;  // zero between launches
  int* next_token;    // where the token goes
  int advance;        // last CTA does seq_len[seq] += 1
  unsigned* guard;
  int fail_token;     // nonzero: a NaN logit or a timed-out wait makes the token -1
};
constexpr int kGemvKcMax = 10;

// Every kernel of the step asks for the largest shared-memory carveout, so
// consecutive kernels never make an SM reconfigure its L1/shared split (which
// needs the SM drained) and can be resident together under programmatic
// dependent launch.
template <typename Kernel>
inline cudaError_t set_kernel_smem(Kernel kernel, int dyn_bytes) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              static_cast<int>(cudaSharedmemCarveoutMaxShared));
}
constexpr int kGemvThreads = 256;

// chooses R / nslice / kc / stages for a weight shape; false if unsupported
bool gemv_plan(GemvArgs& a, int wbytes, int epi, size_t smem_budget);
cudaError_t gemv_init_attrs();
cudaError_t launch_gemv(const GemvArgs& a, int wbytes, int epi, int grid, cudaStream_t s, bool pdl);
size_t gemv_smem_bytes(const GemvArgs& a);

// ---------------------------------------------------------------------------
// packed streaming GEMV (the decode hot path): W is stored pair-interleaved,
// [ceil(N/2) pairs][CT chunks][2 rows][CH elements], CH = 512 bytes / element
// size, zero-padded to whole chunks and pairs, so that any run of (pair, chunk)
// units is one contiguous byte range (1 KB per unit)
// ---------------------------------------------------------------------------
struct PackedGemvArgs {
  const void* Wp;
  int N, K, CT;
  const float* x;    // [K] fp32
  const void* gain;  // [K] norm gain (weight dtype) or null
  int groups;
  float eps;
  int SU;  // units (1 KB) per slot = bytes of one bulk copy / 1024
  int NS;  // slots per warp ring
  uint32_t x_bytes;
  // epilogue (as GemvArgs)
  float* out;
  const float2* rope;
  int cap;
  int* seq_len;
  int seq;
  int head_dim;
  int n_rot_heads;
  float* logits;
  float* part_val;
  int* part_idx;
  unsigned* counter;
  int* next_token;
  int advance;
  unsigned* guard;
};
constexpr int kPackedThreads = 256;
constexpr int kPackedWarps = 8;
constexpr int kPackedMaxSlots = 8;

// bytes of the packed copy of an [N, K] matrix
size_t packed_bytes(int N, int K, int wbytes);
bool packed_plan(PackedGemvArgs& a, int wbytes, size_t smem_budget, int max_slots);
int packed_grid(int N, int sms);
cudaError_t packed_init_attrs();
cudaError_t launch_packed_gemv(const PackedGemvArgs& a, int wbytes, int epi, int grid, cudaStream_t s, bool pdl);
size_t packed_smem_bytes(const PackedGemvArgs& a);

// pack kernels: logical row R of the packed matrix comes from
//   PACK_PLAIN:  src0 row R
//   PACK_QKV:    heads of [src0 (nq heads); src1 (nkv); src2 (nkv)], rows of
//                each head ordered (0, d/2), (1, d/2 + 1), ... (split-half RoPE pairs)
//   PACK_GATEUP: row 2i = src0 row i, row 2i + 1 = src1 row i
enum PackMode : int { PACK_PLAIN = 0, PACK_QKV = 1, PACK_GATEUP = 2 };
// Layouts of quantized packed matrices (described with kWfmtQ4): plain
// row-major codes, pair units, or 16-row tile units for the tensor cores.
enum { LAYOUT_PLAIN = 0, LAYOUT_PAIRS = 1, LAYOUT_TILES = 2 };
// fp8 (E4M3) rows with one fp32 scale per row from bf16 sources (the row mapping
// of launch_pack); LAYOUT_PAIRS: the pair/chunk layout with 512 codes per
// chunk; LAYOUT_TILES: fp8 tile units; LAYOUT_PLAIN: row-major codes [N][K].
// scales get one entry per (padded) row.
cudaError_t launch_quant_pack(uint8_t* dst, float* scales, const void* src0, const void* src1, const void* src2,
                              int mode, int N, int K, int nq, int nkv, int d, int layout, cudaStream_t s);
size_t f8_packed_bytes(int N, int K, bool tiles);
// int4 block quantization (symmetric, codes in [-7, 7], s = max|w| / 7 per 64
// weights of a row, nearest with ties to even) of bf16 sources, with the row
// mapping of launch_pack.  layout LAYOUT_PAIRS / LAYOUT_TILES: the int4 pair or tile
// units (described with kWfmtQ4; dst only, scales unused; tiles: dst is
// cleared first); LAYOUT_PLAIN: int8 codes [N][K] and scales [N][ceil(K / 64)].
cudaError_t launch_q4_pack(uint8_t* dst, float* scales, const void* src0, const void* src1, const void* src2,
                           int mode, int N, int K, int nq, int nkv, int d, int layout, cudaStream_t s);
size_t q4_packed_bytes(int N, int K, bool tiles);
// int4 packed weights (pair or tile units) as bf16 hi / lo halves of code * scale
// in the bf16 packed layout (packed_bytes(N, K, 2) bytes each), for the
// tensor-core prefill
cudaError_t launch_q4_dequant(void* hi, void* lo, const uint8_t* src, int N, int K, bool tiles, cudaStream_t s);
// The fp8 codes of a packed matrix (pair units of 512 per chunk and row, or
// tile units) as bf16 values (exact: every E4M3 value is a bf16 value) in the
// bf16 packed layout (256 per chunk and row).
cudaError_t launch_f8_expand(void* dst, const uint8_t* src, int N, int K, bool tiles, cudaStream_t s);
cudaError_t launch_pack(void* dst, const void* src0, const void* src1, const void* src2, int mode, int N, int K,
                        int wbytes, int nq, int nkv, int d, cudaStream_t s);

// ---------------------------------------------------------------------------
// split-K flash-decode GQA attention with the KV append of the new token
// ---------------------------------------------------------------------------
struct AttnArgs {
  const void* kc;  // K cache of this layer: [batch][nkv][cap][D] in the KV dtype
  const void* vc;
  void* kc_w;  // same pointers, written at row pos
  void* vc_w;
  void* ks;  // int8 scales [batch][nkv][cap] fp16 (null otherwise)
  void* vs;
  int cap;
  const float* qkv;  // [batch][qkv_stride] fp32: q (nq*D, rotated) | k (nkv*D, rotated) | v (nkv*D)
  int qkv_stride;
  // non-null: qkv holds the QKV GEMM's packed rows instead (each head's dims
  // as pairs (i, i + D/2) side by side, not rotated) and the kernel rotates q
  // and k at the token's position with this table [cap][D/2] (cos, sin)
  const float2* rope;
  int nq, nkv;
  const int* seq_len;
  int seq0;             // sequences seq0 .. seq0 + gridDim.z - 1
  float* out;           // [batch][nq*D] fp32 (nullable when out_hi is given)
  __nv_bfloat16* out_hi;  // nullable: the output also as bf16 hi = bf16(o), lo = bf16(o - hi)
  __nv_bfloat16* out_lo;  //   (the activations of a tensor-core GEMM), [batch][nq*D]
  float scale;          // 1/sqrt(D)
  uint32_t slot_bytes;  // one warp's tile slot
  unsigned* guard;
  // block mode (non-zero): every slot b is a query of sequence block_seq at
  // position pos_base + b whose K/V row is already in the cache (a short
  // causal block appended by the prefill path); nothing is written to the cache
  int block_mode;
  int block_seq;
  int pos_base;
  const int* pos_base_dev;  // block mode: read pos_base from device memory (nullable)
  // fp16 caches: host copies of the CUtensorMaps of this layer's K and V
  // (attn_encode_kv); when both are set the tensor-core kernel runs
  const void* map_k;
  const void* map_v;
};
constexpr int kAttnThreads = 128;     // 4 warps: three CTAs (12 warps) share an SM
constexpr int kAttnTK = 32;          // keys per tile; a warp reads one tile at a time
constexpr int kAttnMaxCluster = 16;  // key-range splits of one KV head = one thread-block cluster

bool attn_supported(int head_dim, int rep, int kv_dtype);
size_t attn_slot_bytes(int head_dim, int kv_dtype);
cudaError_t attn_init_attrs();
// largest cluster (<= limit) of this attention kernel that fits the GPU; 0 on error
int attn_max_cluster(int head_dim, int rep, int kv_dtype, int limit);
int attn_ctas_per_sm(int head_dim, int rep, int kv_dtype);  // resident CTAs of the attention kernel per SM
cudaError_t launch_attn(const AttnArgs& a, int head_dim, int rep, int kv_dtype, int nsplit, int batch,
                        cudaStream_t s, bool pdl);
// the tensor-core attention (fp16 caches): shapes it covers, and the tensor map of
// one layer's K or V cache, [rows][head_dim] fp16 (rows = batch * n_kv_heads * cap)
bool attn_tc_supported(int head_dim, int rep);
bool attn_encode_kv(void* map, const void* base, long long rows, int head_dim);

// ---------------------------------------------------------------------------
// persistent batch-1 decode step (one cooperative launch per token)
// ---------------------------------------------------------------------------
struct LayerPtrs {
  const void* wqkv;  // packed
  const void* wo;
  const void* wgu;
  const void* wdown;
  const void* attn_norm;
  const void* mlp_norm;
  void* kc;  // K/V cache of the layer [batch][nkv][cap][D] and int8 scales
  void* vc;
  void* ks;
  void* vs;
};
struct MegaGemv {
  int CT;  // 512-byte chunks per row (the packed layout)
};
// ---- sampling (k2_sample.cu) -------------------------------------------------
constexpr int kSampleThreads = 256;
constexpr int kSampleBins = 2048;     // radix digits of 11 bits
constexpr int kSampleCtaMax = 64;     // CTAs per row
constexpr int kSampleBarBytes = 256;  // the grid-barrier counter, before the rows' scratch
constexpr int kSampleSmemMax = 160 * 1024;  // z of one CTA's vocabulary slice
struct SampleArgs {
  const float* logits;  // row r at logits + r * ld
  size_t ld;
  int vocab;
  const int* seen;      // row r's seen ids at seen + r * seen_stride (nullable: no penalty)
  int seen_stride;
  const int* seen_len;  // [rows]
  const int* counter;   // [rows]: Philox counter word 0 (the position the token takes)
  int first_seq;        // counter word 1 = first_seq + r
  int* next;            // [rows]: the drawn ids
  float temperature, top_p, min_p, penalty;
  int top_k;
  uint32_t key0, key1;  // the seed
  uint8_t* scratch;     // kSampleBarBytes + rows * row_bytes, zeroed by launch_sample
  size_t row_bytes;
  int ctas_per_row;
  unsigned* guard;
};
int sample_ctas_per_row(int rows, int vocab);  // 0: the vocabulary does not fit
size_t sample_row_bytes(int vocab);
cudaError_t launch_sample(const SampleArgs& a, int rows, cudaStream_t s);
cudaError_t launch_philox(uint32_t first, int n, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1,
                          uint32_t* out, cudaStream_t s);

struct MegaArgs {
  // fp8 weights: one fp32 scale per packed row of each matrix (null otherwise);
  // layer l's scales at sc_* + l * ss_*
  const float* sc_qkv;
  const float* sc_o;
  const float* sc_gu;
  const float* sc_down;
  const float* sc_lm;
  size_t ss_qkv, ss_o, ss_gu, ss_down;
  int* hist;  // token history [seq][cap]: the step records its input token at its position (nullable)
  const LayerPtrs* layers;  // device table, n_layers entries (read once per launch: the norm gains)
  int n_layers;
  // packed weights and KV cache of layer l = base + l * stride (bytes)
  const uint8_t* w_qkv;
  const uint8_t* w_o;
  const uint8_t* w_gu;
  const uint8_t* w_down;
  unsigned long long ws_qkv, ws_o, ws_gu, ws_down;
  uint8_t* kc;
  uint8_t* vc;
  uint8_t* ks;  // int8 KV scales (null otherwise)
  uint8_t* vs;
  unsigned long long s_kv, s_sc;
  const void* embed;
  const void* lm_head;  // packed
  const void* final_norm;
  int hidden, vocab, nq, nkv, groups, inter;
  float eps, scale;
  MegaGemv g_qkv, g_o, g_gu, g_down, g_lm;
  int cap, nsplit;
  const float2* rope;
  int* seq_len;
  int seq;
  const int* token_in;
  int* token_out;
  float* logits;     // optional
  float* x_ext;      // layers-only step: the hidden vector in and out; else null
  float* x_out;      // plain fp32 copy of the residual leaving the last layer
  int head;          // 1: final norm + lm_head + argmax after the layers
  // activations as (value, tag) words: a consumer waits for the tag of the
  // phase that writes them
  unsigned long long* t_resid;
  unsigned long long* t_qkv;
  unsigned long long* t_attn;
  unsigned long long* t_act;
  unsigned long long* t_part;  // attention partials [nkv * nsplit][rep * (d + 2)], tagged
  float* am_val;     // per-CTA argmax partials
  int* am_idx;
  unsigned* end_count;
  unsigned* epoch;   // launches so far (tags are derived from it)
  unsigned* guard;
  // how long a wait for another CTA's tagged words may last (waits for this
  // CTA's own bulk copies keep kWaitLimitNs: a copy must land before its CTA exits)
  unsigned long long poll_limit_ns;
  // >= 0: phase stall_phase waits for a tag that no phase writes, so its
  // waits run out (tests of the timeout path); -1 otherwise
  int stall_phase;
  // at the start of every phase whose kind j (0 QKV .. 4 down, 5 lm_head) has
  // bit j set in l2_mask, each warp asks L2 for its next l2_ahead slots beyond
  // those already in flight, so that they stream while the phase waits for
  // its input
  int l2_ahead;
  int l2_mask;
  // measurement: when set, thread 0 of every CTA stamps %globaltimer (ns) at
  // trace[(q * gridDim + cta) * 4 + k] for phase q: k = 0 phase start, 1 input
  // ready, 2 weight / K-V slots consumed, 3 phase end
  unsigned long long* trace;
};
// fp16 caches of a head_dim that is a multiple of 64: the persistent step
// reads K and V tiles through these tensor maps ([layer][rows][head_dim] fp16,
// boxes of 64 dims x kMegaTK rows, 128-byte swizzle); zero otherwise
struct KvMaps {
  CUtensorMap k, v;
};
constexpr int kMegaThreads = 256;
constexpr int kMegaSlots = 2;                 // ring slots per warp
constexpr int kMegaSlotBytes = 9 * 1024;      // one bulk copy: 9 packed units, or one 16-key K/V tile
constexpr int kMegaRingBytes = 8 * kMegaSlots * kMegaSlotBytes;
constexpr int kMegaXBytes = 40 * 1024;        // the normalised input vector (K <= 10240 at bf16)
constexpr int kMegaGainBytes = 8 * 1024;      // one norm gain (hidden x weight bytes); two buffers
constexpr int kMegaSmemBytes = kMegaRingBytes + kMegaXBytes + 2 * kMegaGainBytes;
constexpr int kMegaTK = 16;                   // keys per attention tile (at most)
constexpr unsigned kMegaPollSleepNs = 0;      // pause between rounds of a tag poll
constexpr int kMegaPairsMax = 64;             // row pairs of one CTA in the QKV / residual phases
constexpr int kMegaSplitMax = 64;             // key splits per KV head in the attention phase
constexpr int kMegaTagShift = 10;
constexpr int kMegaMaxLayers = 64;            // norm-gain pointers kept in shared memory
// tag = (epoch + 1) << kMegaTagShift | phase: at most 1023 phases

// Packed weight formats of the persistent step, the key that picks its
// kernel: the bytes of one weight for fp32 (4), bf16 (2) and fp8 E4M3 (1), or
// kWfmtQ4 for int4 codes with one fp32 scale per 64 weights of a row.
//
// fp8 and int4 matrices come in two layouts.  Pair units (QKV, o_proj, down):
// a 512-weight chunk of both rows of a pair -- fp8: row 0's 512 codes, then
// row 1's; int4: row 0's 256 bytes of codes (the code of weight 2i in the low
// nibble of byte i), row 1's, then row 0's 8 block scales and row 1's.  Tile
// units (gate/up and lm_head, the tiled_kind kinds, whose many rows keep
// 16-row ownership balanced over the SMs), for the tensor cores: one unit
// holds one 64-weight block of 16 packed rows (8 row pairs, a "tile"), units
// ordered tile-major, block minor.  Tile row m (the A row of mma.sync
// m16n8k16) is packed row 2 (m % 8) + m / 8 of the tile, so rows m and m + 8
// are the two rows of pair m % 8.
//
// fp8 tile unit (1024 bytes): for MMA j (weights 16j .. 16j + 15 of the
// block), lane 4 g + t's 8 codes -- rows g, g, g + 8, g + 8 at positions
// 2t, 2t + 1, then the same rows at 2t + 8, 2t + 9 -- sit at byte
// 512 (j / 2) + 16 lane + 8 (j % 2); each code pair converts to one A fragment
// register (fp8x2 -> f16x2, exact).
//
// int4 tile unit: bytes 0..511: 32 lanes x 4 words, word j (MMA j: weights 16j ..
// 16j + 15 of the block) of lane 4 g + t holding the eight nibbles (code + 8)
// of rows g and g + 8 at block positions 16j + {2t, 2t + 1, 2t + 8, 2t + 9},
// at bit 4 (m >= 8) + 8 (position >= 2t + 8) + 16 (odd position) -- so that
// a nibble pair OR-ed into fp16 1024 and one fp16 add (or fma) give an A
// fragment register of exact codes.  Bytes 512..575: the 16 rows' fp32 block
// scales, pair p's two at 512 + 8 p.
constexpr int kWfmtQ4 = 5;
constexpr int kQ4Block = 64;
constexpr int kQ4Chunk = 512;  // weights of a row handled by one CTA of the quantizer
constexpr int kQ4Unit = 576;
constexpr int kQ4GroupRows = 16;
// GEMV kinds of the persistent step (0 QKV, 1 o_proj, 2 gate/up, 3 down,
// 4 lm_head) whose fp8 and int4 weights use the tile layout
__host__ __device__ constexpr bool tiled_kind(int kind) { return kind == 2 || kind == 4; }

bool mega_supported(int wfmt, int head_dim, int rep, int kv_dtype);
cudaError_t mega_init_attrs(int wfmt, int head_dim, int rep, int kv_dtype);
int mega_max_grid(int wfmt, int head_dim, int rep, int kv_dtype);  // 0: cannot run
cudaError_t launch_mega(const MegaArgs& a, const KvMaps& maps, int wfmt, int head_dim, int rep, int kv_dtype, int grid,
                        cudaStream_t s);
// the persistent step runs its attention on the tensor cores (and needs KvMaps)
bool mega_tc_attention(int head_dim, int kv_dtype);
// tensor map of every layer's K or V cache: [layers][rows][head_dim] fp16, layer
// l at base + l * layer_stride bytes, boxes of 64 dims x box_rows rows
bool attn_encode_kv_layers(void* map, const void* base, long long rows, int head_dim, int layers,
                           unsigned long long layer_stride, int box_rows);

// ---------------------------------------------------------------------------
// small kernels
// ---------------------------------------------------------------------------
// hist (nullable): the token of block b is recorded at hist[b * hist_stride + pos[b]]
cudaError_t launch_embed(const void* E, int wbytes, int vocab, int hidden, const int* tokens, int batch,
                         float* resid, unsigned* guard, int* hist, int hist_stride, const int* pos, cudaStream_t s,
                         bool pdl);
cudaError_t launch_rope_table(float2* tab, int cap, int head_dim, double theta, cudaStream_t s);
cudaError_t launch_repack_qkv(void* dst, const void* wq, const void* wk, const void* wv, int wbytes, int nq,
                              int nkv, int d, int hidden, cudaStream_t s);
cudaError_t launch_repack_gateup(void* dst, const void* wg, const void* wu, int wbytes, int inter, int hidden,
                                 cudaStream_t s);
cudaError_t launch_advance(int* seq_len, int seq0, int batch, cudaStream_t s, bool pdl);

// ---- prefill: tensor-core GEMMs (k2_tcgemm.cu) and the row-wise kernels (k2_prefill.cu)
enum { TC_STORE = 0, TC_RESID = 1, TC_SWIGLU = 2 };
struct TcGemmArgs {
  int N;       // weight rows (packed order)
  int K;       // reduction length
  int T;       // tokens
  int ksteps;  // 64-element K steps over the packed chunks: 4 * ceil(K / 256)
  int mode;    // TC_STORE: out[t][row] = acc; TC_RESID: out[t][row] += acc;
               // TC_SWIGLU: rows (2p, 2p+1) -> silu(gate) * up -> out_hi/out_lo[t][p]
  int ldo;     // row stride of the output (elements)
  int tile_tokens;  // 128 (prefill) or 16 (batched decode): must match the activation maps
  int splits;  // split-K: blockIdx.z takes K steps [ksteps*z/splits, ksteps*(z+1)/splits) and
               // adds its partial with atomicAdd (TC_STORE / TC_RESID only; 1 = no split)
  int f16;     // 1: fp16 operands (the weights' fp16 copy, single fp16 activations: no low-half map);
               // TC_SWIGLU then writes fp16 into out_hi
  int whole;   // persistent kernel: 1 = each CTA takes whole tiles (b, b + grid, ...) and the
               // epilogue stores / adds / applies SwiGLU; 0 = stream-K shares with atomicAdd
  float* out;
  __nv_bfloat16* out_hi;
  __nv_bfloat16* out_lo;   // TC_SWIGLU: nullable (only the high half is written)
  unsigned* guard;
  const float* row_scale;  // non-null: each row's accumulator is multiplied by row_scale[row] first
};
constexpr int kTcMapBytes = 128;  // one CUtensorMap
bool tc_encode_weight(void* map, const void* packed, int N, int K);  // bf16 packed weights
bool tc_encode_act(void* map, const void* buf, int rows, int K, int tile_tokens);  // bf16 [rows][K]
cudaError_t tc_gemm_init_attrs();
// mapXl (the activations' low halves) null: one MMA per K step on the high
// halves alone (tile_tokens 128 only).  mapWl (nullable; tile_tokens 128 with
// mapXl): the weights' low halves, a third MMA per K step (w_lo . x_hi).
cudaError_t launch_tc_gemm(const void* mapW, const void* mapWl, const void* mapXh, const void* mapXl,
                           const TcGemmArgs& a, cudaStream_t s);
// persistent variant, `ctas` CTAs: stream-K (whole = 0; TC_STORE into a zeroed target or TC_RESID)
// or whole tiles (whole = 1; any mode, tile_tokens 128 or 16).
// pdl: programmatic dependent launch; the first weight stages are requested before
// the kernel waits for its predecessor (weights never depend on an earlier kernel)
cudaError_t launch_tc_gemm_sk(const void* mapW, const void* mapWl, const void* mapXh, const void* mapXl,
                              const TcGemmArgs& a, int ctas, cudaStream_t s, bool pdl = false);
// Causal prefill attention on the tensor cores (tcgen05, fp16 caches): the n
// query tokens of a block at positions pos0 .. pos0 + n - 1 (Q [n][nq * D] fp32,
// rotated) against every cached key of their sequence up to their own position,
// through `maps` (the K and V caches of every layer, boxes of 64 dims x 64 rows);
// the attention output goes to oh / ol [n][nq * D] as bf16 hi / lo halves.
// split: queries and probabilities enter the MMAs as fp16 hi + lo halves (two
// MMAs each), else as single fp16 values; ol (nullable) receives the output's
// bf16 low halves.
struct PrefillAttnArgs {
  const float* Q;
  __nv_bfloat16* oh;
  __nv_bfloat16* ol;
  int n, nq, nkv;
  int pos0;
  int head_row0;  // cache row of key 0 of KV head 0 of the sequence (KV head g at + g * cap)
  int cap;
  int layer;
  float scale;
  unsigned* guard;
  int split;
  int f16out;  // 1: the output is written as single fp16 into oh (ol unused)
};
bool prefill_attn_tc_supported(int head_dim, int rep);
cudaError_t prefill_attn_tc_init_attrs();
cudaError_t launch_prefill_attn_tc(const KvMaps& maps, const PrefillAttnArgs& a, int head_dim, int rep,
                                   cudaStream_t s);
bool prefill_attn_supported(int head_dim, int rep);
cudaError_t prefill_init_attrs();
// hist (nullable): row t's token is recorded at hist[t * hist_stride + pos[t]], or at
// hist[pos0 + t] when pos is null (pos0 read from pos0_dev when that is not null)
cudaError_t launch_embed_rows(const int* tokens, int n, const void* E, int wbytes, float* X, int H, int vocab,
                              unsigned* guard, int* hist, int hist_stride, const int* pos, int pos0,
                              const int* pos0_dev, cudaStream_t s, bool pdl = false);
// GroupedRMSNorm rows -> bf16 hi/lo (f16: single fp16 into oh, ol unused, a value
// beyond the fp16 range raises GUARD_RANGE in guard); zero (nullable, zero_floats a
// multiple of 4, 16-byte aligned): extra CTAs clear it (the output of the GEMM that
// follows); copy (nullable): the rows of X are also copied there
cudaError_t launch_norm_rows(const float* X, int n, const void* gain, int wbytes, __nv_bfloat16* oh,
                             __nv_bfloat16* ol, int H, int groups, float eps, cudaStream_t s, bool pdl = false,
                             float* zero = nullptr, size_t zero_floats = 0, float* copy = nullptr, bool f16 = false,
                             unsigned* guard = nullptr);
// n bf16 values -> fp16 (round to nearest even; exact in fp16's normal range); a value
// beyond +-65504 is clamped there and raises GUARD_RANGE in guard.  n a multiple of 8,
// both buffers 16-byte aligned.
cudaError_t launch_bf16_to_f16(__half* dst, const __nv_bfloat16* src, size_t n, unsigned* guard, cudaStream_t s);
// pos0_dev (nullable): read the first position from device memory instead of pos0
cudaError_t launch_rope_append(const float* qkv, float* Q, const float2* rope, int kv_dtype, void* kc, void* vc,
                               void* ks, void* vs, int n, int nq, int nkv, int D, int pos0, const int* pos0_dev,
                               size_t head_row0, int cap, cudaStream_t s, bool pdl = false);
cudaError_t launch_prefill_attn(const float* Q, int kv_dtype, const void* kc, const void* vc, const void* ks,
                                const void* vs, __nv_bfloat16* oh, __nv_bfloat16* ol, int n, int nq, int nkv, int D,
                                int pos0, size_t head_row0, int cap, float scale, cudaStream_t s);
cudaError_t launch_advance_by(int* seq_len, int seq, int n, cudaStream_t s);
cudaError_t launch_swiglu_rows(const float* gu, __nv_bfloat16* oh, __nv_bfloat16* ol, int rows, int I, cudaStream_t s,
                               bool pdl = false);
cudaError_t launch_rows_hilo(const float* x, __nv_bfloat16* oh, __nv_bfloat16* ol, int rows, int K, cudaStream_t s,
                             bool pdl = false);
cudaError_t launch_argmax_rows(const float* logits, int rows, int V, int* next, float* part_val, int* part_idx,
                               int part_stride, unsigned* guard, cudaStream_t s, bool pdl = false);
cudaError_t misc_init_attrs();

}  // namespace k2
