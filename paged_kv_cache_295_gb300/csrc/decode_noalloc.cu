// paged_attention_decode_noalloc: the decode entry point for callers that are
// not allowed to allocate device memory.
//
// The split-KV partials that paged_attention_decode keeps in a caller-supplied
// workspace live here in a fixed array compiled into the library instead, so
// a caller only passes its inputs and outputs.  This is for code that runs
// where an allocation is not an option: a plug-in inside a host program that
// owns every device allocation itself, a runtime that plans all of its memory
// once at start-up and forbids allocating on the per-token path, or a caller
// that must not trigger the device-wide synchronisation an allocation can
// cause.
//
// Costs and rules of the fixed array:
//  * every GPU that loads this library holds PKV_NOALLOC_SCRATCH_BYTES of
//    device memory for it until the process exits;
//  * a request whose partials would need more returns PKV_ERR_SCRATCH_LIMIT
//    before anything runs;
//  * all calls on a device share the one array: two calls whose kernels
//    overlap on the GPU (different streams, no ordering between them) race on
//    it and may corrupt each other's outputs.  Calls on one stream are safe;
//  * the array keeps whatever the previous call left in it.  Nothing has to
//    start at zero: each call writes every partial before it reads it.
//  * The first call on each device looks up the array's device address
//    (cudaGetSymbolAddress with that device current) and remembers it with
//    the unique id of the context it belongs to; make that first call before
//    any stream capture begins.  When a later call finds another context
//    current on that device (the old one was destroyed, e.g. by
//    cudaDeviceReset, and the library's module loaded again), it looks the
//    address up again, so that call too should come before any capture.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace pkv {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  unsigned long long ctx_id;   // the context the address belongs to
  void* addr;
};
ScratchAddr g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Unique id of the calling thread's current context, or 0 when there is none
// yet (the driver's functions are reached through the runtime, so the library
// links no libcuda).
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    cudaGetLastError();
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_decode_scratch on the current device.  In host code the
// symbol's name is only a host-side handle, never a device pointer, so the
// kernels get the address cudaGetSymbolAddress returns.  It is looked up once
// per device and context: again only when the device's context has changed.
pkv_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = current_context_id();
  ScratchAddr& c = g_scratch[dev];
  if (c.addr == nullptr || id == 0 || id != c.ctx_id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
    c.addr = p;
    c.ctx_id = current_context_id();   // the lookup made the context current if it was not
  }
  *out = c.addr;
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status paged_attention_decode_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq,
    int32_t max_context_len, float scale, int32_t q_dtype, int32_t kv_dtype, const float* k_scale,
    const float* v_scale, float* out, int32_t partition_tokens, int32_t* device_status,
    pkv_stream_t stream) {
  const size_t need = paged_attention_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                      head_dim, max_context_len, partition_tokens);
  if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const pkv_status st = pkv::scratch_address(&scratch);
  if (st != PKV_OK) return st;
  return paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                max_blocks_per_seq, max_context_len, scale, q_dtype, kv_dtype,
                                k_scale, v_scale, out, scratch, PKV_NOALLOC_SCRATCH_BYTES,
                                partition_tokens, device_status, stream);
}
