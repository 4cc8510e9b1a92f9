// decode_noalloc.cu -- decode attention for callers that cannot allocate GPU
// memory.  Plugin hosts of inference engines often hand a kernel only its
// input and output buffers, and some serving loops cannot afford the device
// synchronisation that cudaMalloc implies; such callers have no way to provide
// the split-K workspace that kvarn_decode_attention asks for.  This entry
// point keeps that scratch in a fixed-size array inside the library instead.
//
// The array lives in this file as a static __device__ variable, so every GPU
// that loads the library holds KVARN_NOALLOC_SCRATCH_BYTES of it until the
// process exits.  Host code cannot use the array's name as a device address:
// on each device the first call looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it.  That first
// call per device should therefore be made before any stream capture begins.
// The cache is keyed by the device's current context as well: after a
// cudaDeviceReset the module is loaded afresh and the array may move, so a
// call in a new context looks the address up again (and should, like the
// first call, come before any stream capture).
// All calls share the one array, which keeps the contents of the last call:
// the ticket counters that must start at zero are cleared on every call that
// merges splits through them, and calls whose executions overlap on the GPU
// race on the array.
#include <mutex>

#include "kvarn_internal.cuh"

namespace kvarn {
namespace {

constexpr size_t kScratchBytes = KVARN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};   // context id the address belongs to

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Process-unique id of the current context (0 when there is none yet or the
// driver cannot say).  Ids are never reused, unlike context handles.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_scratch in the current device's current context,
// looked up once per (device, context).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVARN_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return KVARN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long ctx = current_context_id();
  if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* ptr = nullptr;
    // initialises the context if the runtime has not yet done so
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || !ptr) return KVARN_ERR_LAUNCH;
    g_scratch_addr[dev] = ptr;
    g_scratch_ctx[dev] = current_context_id();
  }
  *out = g_scratch_addr[dev];
  return KVARN_OK;
}

}  // namespace
}  // namespace kvarn

using namespace kvarn;

extern "C" int kvarn_decode_attention_noalloc(const kvarn_config_t* cfg, const void* q,
                                              const void* pool, int64_t num_pages,
                                              const int32_t* block_table, int max_blocks,
                                              const int32_t* seq_lens, int batch, int max_seq,
                                              const void* tail_k, const void* tail_v,
                                              float softmax_scale, void* out, int32_t* status,
                                              kvarn_stream_t stream) {
  // the same host checks as kvarn_decode_attention, so a rejected call leaves
  // the scratch and the stream untouched
  int rc = kvarn_config_validate(cfg);
  if (rc != KVARN_OK) return rc;
  if (batch < 0 || max_seq < 0 || max_blocks < 0 || num_pages < 0) return KVARN_ERR_INVALID_ARG;
  if (batch == 0) return KVARN_OK;
  if (!q || !seq_lens || !tail_k || !tail_v || !out) return KVARN_ERR_INVALID_ARG;
  if (max_seq >= kT && (!pool || !block_table || num_pages <= 0 || max_blocks < max_seq / kT))
    return KVARN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool) || !aligned16(tail_k) || !aligned16(tail_v) ||
      !aligned16(out))
    return KVARN_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return KVARN_ERR_INVALID_ARG;
  if (batch > 65535 || cfg->num_kv_heads > 65535) return KVARN_ERR_UNSUPPORTED;

  const int sms = device_sm_count();
  if (sms <= 0) return KVARN_ERR_LAUNCH;
  const DecodePlan p = decode_plan(batch, cfg->num_q_heads, cfg->num_kv_heads, max_seq, sms,
                                     cfg_fmt(cfg));
  const size_t need = p.part_bytes + p.count_bytes;
  if (need > kScratchBytes) return KVARN_ERR_WORKSPACE;   // beyond the built-in scratch
  void* ws = nullptr;
  if (need > 0) {
    rc = scratch_address(&ws);
    if (rc != KVARN_OK) return rc;
    // the arrival tickets must start at zero whatever an earlier call left;
    // a plan that merges its splits inside a thread-block cluster never reads
    // them, so it needs no clearing
    if (!p.cluster &&
        cudaMemsetAsync(static_cast<unsigned char*>(ws) + p.part_bytes, 0, p.count_bytes,
                        (cudaStream_t)stream) != cudaSuccess)
      return KVARN_ERR_LAUNCH;
  }
  return kvarn_decode_attention(cfg, q, pool, num_pages, block_table, max_blocks, seq_lens,
                                batch, max_seq, tail_k, tail_v, softmax_scale, out, ws, need,
                                status, stream);
}
