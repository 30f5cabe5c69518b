// k2_greedy_head_noalloc: the greedy head (final GroupedRMSNorm + lm_head
// GEMV + first-index argmax) for callers that cannot allocate device memory.
//
// Who needs it: code that runs inside a host runtime which owns every device
// buffer and hands out no allocator (an inference-server plugin with a
// pre-planned memory arena, for instance), and code on a latency-critical path
// that must not call cudaMalloc because cudaMalloc may synchronise the whole
// device.  Such a caller has its own hidden state and weights and wants a
// token, but cannot provide the per-CTA scratch that the lm_head kernel uses
// to combine its partial maxima.
//
// The scratch lives here instead, in one file-scope device array of fixed
// size that every GPU loading this library keeps until the process exits.
// All calls share it, so calls whose kernels overlap on the GPU (two streams,
// or two host threads) race on it; serialise them.  Each call clears the
// counter and the guard bits it relies on before its kernel runs.
//
// A caller without a context has no k2_sync_status to ask, so a call whose
// logits hold a NaN, or whose kernel gave up on a bounded wait, writes -1 as
// its token instead of an index; every other call writes the first index of
// the maximum logit.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/k2.h"
#include "k2_kernels.h"

namespace {

constexpr int kMaxCtas = K2_NOALLOC_MAX_CTAS;
constexpr int kMaxDevices = 64;

struct HeadScratch {
  float val[kMaxCtas];  // per-CTA best logit
  int idx[kMaxCtas];    // per-CTA index of that logit
  unsigned counter;     // CTAs finished; the kernel's last CTA resets it to 0
  unsigned guard;       // device guard bits (NaN logits, a wait that ran out) of this call
};

static __device__ __align__(256) unsigned char g_head_scratch[sizeof(HeadScratch)];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_head_scratch, per device

}  // namespace

extern "C" k2_status k2_greedy_head_noalloc(const k2_config* cfg, const void* lm_head, const void* final_norm,
                                            const float* d_x, float* d_logits, int32_t* d_token, void* stream) {
  if (!cfg || !lm_head || !final_norm || !d_x || !d_token) return K2_ERR_ARG;
  if (cfg->hidden <= 0 || cfg->vocab <= 0 || cfg->norm_groups <= 0 || cfg->hidden % cfg->norm_groups)
    return K2_ERR_SHAPE;
  if (cfg->weight_dtype != K2_F32 && cfg->weight_dtype != K2_BF16) return K2_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(d_x) % 16 || reinterpret_cast<uintptr_t>(lm_head) % 16 ||
      reinterpret_cast<uintptr_t>(final_norm) % 16)
    return K2_ERR_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return K2_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return K2_ERR_CUDA;

  // one-time set-up per device, with that device current: the device address
  // of the static scratch (host code may not use the symbol itself) and the
  // kernels' shared-memory limits
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_head_scratch) != cudaSuccess || !p) return K2_ERR_CUDA;
      if (k2::gemv_init_attrs() != cudaSuccess) return K2_ERR_CUDA;
      g_scratch_addr[dev] = p;
    }
    base = g_scratch_addr[dev];
  }
  HeadScratch* scr = static_cast<HeadScratch*>(base);

  const int wb = cfg->weight_dtype == K2_BF16 ? 2 : 4;
  k2::GemvArgs a = {};
  a.W = lm_head;
  a.N = cfg->vocab;
  a.K = cfg->hidden;
  a.x = d_x;
  a.gain = final_norm;
  a.groups = cfg->norm_groups;
  a.eps = cfg->eps;
  if (!k2::gemv_plan(a, wb, k2::EPI_ARGMAX, 96 * 1024)) return K2_ERR_UNSUPPORTED;
  int grid = sms;
  if (grid > a.N / a.align) grid = a.N / a.align;
  if (grid < 1) grid = 1;
  if (grid > kMaxCtas) return K2_ERR_WORKSPACE;  // the static scratch holds kMaxCtas partial maxima
  a.logits = d_logits;
  a.part_val = scr->val;
  a.part_idx = scr->idx;
  a.counter = &scr->counter;
  a.next_token = d_token;
  a.advance = 0;  // no sequence state is touched
  a.guard = &scr->guard;
  a.fail_token = 1;  // the caller has no status word to read: a failed call says so in d_token (-1)
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the counter and guard must start at zero (a call cut short could have left them set)
  if (cudaMemsetAsync(&scr->counter, 0, 2 * sizeof(unsigned), s) != cudaSuccess) return K2_ERR_CUDA;
  if (k2::launch_gemv(a, wb, k2::EPI_ARGMAX, grid, s, false) != cudaSuccess) return K2_ERR_CUDA;
  return K2_OK;
}
