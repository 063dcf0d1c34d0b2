// CUDA-graph decode step ("nano-vLLM architecture" section 5: record once,
// replay; batch-size buckets with padding to the nearest larger bucket;
// "TGI architecture" section 5.1: graphs recorded for common batch sizes).
//
// One graph per bucket holds, for every layer, the append of the step's new
// K/V rows and the decode attention (with its split-KV reduce), captured from
// the library's own entry points on a private stream.  A launch pads the rows
// between the batch and the bucket (context 0, slot -1) with one small kernel
// and replays the bucket's graph on the caller's stream.  decode_graph_step_host
// wraps a launch into the per-token call a serving loop makes from host
// memory: block tables straight from the pool into page-locked staging, one
// copy per input buffer, the replay, the output copied back, one stream sync.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>
#include <vector>

#include "common.cuh"

struct pkv_decode_graph {
  pkv_decode_graph_config cfg{};
  std::vector<void*> k_caches, v_caches;
  std::vector<const float*> k_scales, v_scales;
  std::vector<int32_t> buckets;
  std::vector<cudaGraphExec_t> execs;
  int device = 0;
  int32_t* host_meta = nullptr;   // page-locked [Bmax][max_blocks] tables, then [Bmax] lengths
};

namespace pkv {
namespace {

__global__ void pad_rows_kernel(int32_t* context_lens, int64_t* slot_mapping, int32_t from,
                                int32_t to) {
  const int32_t i = from + blockIdx.x * blockDim.x + threadIdx.x;
  if (i < to) {
    context_lens[i] = 0;
    slot_mapping[i] = -1;
  }
}

pkv_status pad_rows(const pkv_decode_graph_config& c, int32_t from, int32_t to, cudaStream_t st) {
  if (to <= from) return PKV_OK;
  const int32_t n = to - from;
  pad_rows_kernel<<<(n + 255) / 256, 256, 0, st>>>(c.context_lens, c.slot_mapping, from, to);
  return cuda_status(cudaGetLastError());
}

// One strided host -> device copy: `rows` rows of `row_bytes`, the source rows
// `src_stride` apart in mapped page-locked host memory, the destination rows
// `dst_stride` apart on the device.
struct StageSeg {
  const uint8_t* src;
  uint8_t* dst;
  int64_t row_bytes, src_stride, dst_stride;
  int32_t rows;
};
constexpr int kStageSegs = 6;
struct StageArgs {
  StageSeg seg[kStageSegs];
};

// The step's inputs gathered in one launch (blockIdx.y = segment): a kernel
// reading host memory over the host link replaces one DMA copy per buffer.
// 16-byte words where the segment's addresses and sizes allow, else 4-byte.
__global__ void stage_inputs_kernel(const StageArgs a) {
  const StageSeg sg = a.seg[blockIdx.y];
  const bool v16 = ((reinterpret_cast<uintptr_t>(sg.src) | reinterpret_cast<uintptr_t>(sg.dst) |
                     static_cast<uintptr_t>(sg.row_bytes) | static_cast<uintptr_t>(sg.src_stride) |
                     static_cast<uintptr_t>(sg.dst_stride)) & 15u) == 0;
  const int64_t unit = v16 ? 16 : 4;
  const int64_t per_row = sg.row_bytes / unit;
  const int64_t total = per_row * sg.rows;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row, k = i % per_row;
    const uint8_t* src = sg.src + r * sg.src_stride + k * unit;
    uint8_t* dst = sg.dst + r * sg.dst_stride + k * unit;
    if (v16)
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    else
      *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
  }
}

// Device address of page-locked host memory, or nullptr when the pointer is
// not mapped (pageable memory, or no mapping): the caller then copies instead.
const uint8_t* mapped(const void* host) {
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, const_cast<void*>(host), 0) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<const uint8_t*>(d);
}

// The step for a batch of B rows: every layer's append and decode (one fused
// call per layer; one launch per layer where the transposed kernel runs).
pkv_status record_step(const pkv_decode_graph& g, int32_t B, cudaStream_t st) {
  const pkv_decode_graph_config& c = g.cfg;
  const int32_t Bmax = g.buckets.back();
  const int64_t q_layer = static_cast<int64_t>(Bmax) * c.num_q_heads * c.head_dim;
  const int64_t kv_layer = static_cast<int64_t>(Bmax) * c.num_kv_heads * c.head_dim;
  const int qb = elem_bytes(c.q_dtype), sb = elem_bytes(c.src_dtype);
  const int32_t max_ctx = c.max_blocks_per_seq * c.block_size;
  for (int32_t l = 0; l < c.num_layers; ++l) {
    const float* ks = g.k_scales.empty() ? nullptr : g.k_scales[l];
    const float* vs = g.v_scales.empty() ? nullptr : g.v_scales[l];
    const pkv_status s = paged_attention_decode_append(
        static_cast<const uint8_t*>(c.q) + l * q_layer * qb,
        static_cast<const uint8_t*>(c.k_new) + l * kv_layer * sb,
        static_cast<const uint8_t*>(c.v_new) + l * kv_layer * sb, c.slot_mapping, c.src_dtype,
        g.k_caches[l], g.v_caches[l], c.block_tables, c.context_lens, B, c.num_q_heads,
        c.num_kv_heads, c.head_dim, c.block_size, c.num_blocks, c.max_blocks_per_seq, max_ctx,
        c.scale, c.q_dtype, c.kv_dtype, ks, vs, c.out + l * q_layer, c.workspace,
        c.workspace_bytes, 0, c.device_status, reinterpret_cast<pkv_stream_t>(st));
    if (s != PKV_OK) return s;
  }
  return PKV_OK;
}

void release(pkv_decode_graph* g) {
  if (!g) return;
  for (cudaGraphExec_t e : g->execs)
    if (e) cudaGraphExecDestroy(e);
  if (g->host_meta) cudaFreeHost(g->host_meta);
  delete g;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status decode_graph_create(const pkv_decode_graph_config* cfg,
                                          pkv_decode_graph** out) {
  using namespace pkv;
  if (!cfg || !out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  const pkv_decode_graph_config& c = *cfg;
  if (c.num_layers <= 0 || c.num_buckets <= 0 || !c.buckets || !c.k_caches || !c.v_caches ||
      !c.q || !c.k_new || !c.v_new || !c.slot_mapping || !c.block_tables || !c.context_lens ||
      !c.out || c.max_blocks_per_seq <= 0 || c.block_size <= 0 || c.head_dim <= 0 ||
      c.num_q_heads <= 0 || c.num_kv_heads <= 0)
    return PKV_ERR_INVALID_ARG;
  if (elem_bytes(c.q_dtype) == 0 || elem_bytes(c.src_dtype) == 0) return PKV_ERR_UNSUPPORTED;
  const bool scaled = c.kv_dtype == PKV_FP8_E4M3 || c.kv_dtype == PKV_INT8;
  if (scaled && (!c.k_scales || !c.v_scales)) return PKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < c.num_buckets; ++i)
    if (c.buckets[i] <= 0 || (i > 0 && c.buckets[i] <= c.buckets[i - 1]))
      return PKV_ERR_INVALID_ARG;
  const int64_t max_ctx = static_cast<int64_t>(c.max_blocks_per_seq) * c.block_size;
  if (max_ctx > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
  const int32_t Bmax = c.buckets[c.num_buckets - 1];
  for (int32_t i = 0; i < c.num_buckets; ++i)   // every bucket's partials fit the workspace
    if (paged_attention_workspace_bytes(c.buckets[i], c.num_q_heads, c.num_kv_heads, c.head_dim,
                                        static_cast<int32_t>(max_ctx), 0) > c.workspace_bytes)
      return PKV_ERR_INVALID_ARG;

  pkv_decode_graph* g = new (std::nothrow) pkv_decode_graph();
  if (!g) return PKV_ERR_HOST_MEMORY;
  try {
    g->cfg = c;
    g->k_caches.assign(c.k_caches, c.k_caches + c.num_layers);
    g->v_caches.assign(c.v_caches, c.v_caches + c.num_layers);
    if (scaled) {
      g->k_scales.assign(c.k_scales, c.k_scales + c.num_layers);
      g->v_scales.assign(c.v_scales, c.v_scales + c.num_layers);
    }
    g->buckets.assign(c.buckets, c.buckets + c.num_buckets);
    g->execs.assign(c.num_buckets, nullptr);
  } catch (const std::bad_alloc&) {
    delete g;
    return PKV_ERR_HOST_MEMORY;
  }
  g->cfg.k_caches = nullptr;   // the copies above are the ones kept
  g->cfg.v_caches = nullptr;
  g->cfg.k_scales = nullptr;
  g->cfg.v_scales = nullptr;
  g->cfg.buckets = nullptr;
  cudaGetDevice(&g->device);
  if (cudaHostAlloc(reinterpret_cast<void**>(&g->host_meta),
                    static_cast<size_t>(Bmax) * (c.max_blocks_per_seq + 1) * sizeof(int32_t),
                    cudaHostAllocDefault) != cudaSuccess) {
    cudaGetLastError();
    g->host_meta = nullptr;
    release(g);
    return PKV_ERR_CUDA;
  }

  cudaStream_t st = nullptr;
  if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    release(g);
    return PKV_ERR_CUDA;
  }
  pkv_status status = PKV_OK;
  // Load every kernel and set its attributes outside any capture: one run per
  // bucket with all rows padded (nothing appended, outputs 0).
  status = pad_rows(g->cfg, 0, Bmax, st);
  for (int32_t i = 0; status == PKV_OK && i < c.num_buckets; ++i)
    status = record_step(*g, g->buckets[i], st);
  if (status == PKV_OK && cudaStreamSynchronize(st) != cudaSuccess) status = PKV_ERR_CUDA;
  for (int32_t i = 0; status == PKV_OK && i < c.num_buckets; ++i) {
    cudaGraph_t graph = nullptr;
    if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      status = PKV_ERR_CUDA;
      break;
    }
    const pkv_status rs = record_step(*g, g->buckets[i], st);
    const cudaError_t ec = cudaStreamEndCapture(st, &graph);
    if (rs != PKV_OK || ec != cudaSuccess || !graph) {
      status = rs != PKV_OK ? rs : PKV_ERR_CUDA;
      if (graph) cudaGraphDestroy(graph);
      break;
    }
    const cudaError_t ei = cudaGraphInstantiate(&g->execs[i], graph, 0);
    cudaGraphDestroy(graph);
    if (ei != cudaSuccess) {
      g->execs[i] = nullptr;
      status = PKV_ERR_CUDA;
      break;
    }
  }
  if (status == PKV_OK && cudaStreamSynchronize(st) != cudaSuccess) status = PKV_ERR_CUDA;
  cudaStreamDestroy(st);
  if (status != PKV_OK) {
    cudaGetLastError();
    release(g);
    return status;
  }
  *out = g;
  return PKV_OK;
}

extern "C" pkv_status decode_graph_launch(pkv_decode_graph* g, int32_t batch, int32_t* bucket_out,
                                          pkv_stream_t stream) {
  using namespace pkv;
  if (!g || batch <= 0 || batch > g->buckets.back()) return PKV_ERR_INVALID_ARG;
  const auto it = std::lower_bound(g->buckets.begin(), g->buckets.end(), batch);
  const size_t i = static_cast<size_t>(it - g->buckets.begin());
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const pkv_status s = pad_rows(g->cfg, batch, *it, st);
  if (s != PKV_OK) return s;
  if (cudaGraphLaunch(g->execs[i], st) != cudaSuccess) return PKV_ERR_CUDA;
  if (bucket_out) *bucket_out = *it;
  return PKV_OK;
}

extern "C" void decode_graph_destroy(pkv_decode_graph* g) { pkv::release(g); }

extern "C" pkv_status decode_graph_step_host(pkv_decode_graph* g, const pkv_pool* pool,
                                             const int64_t* seq_ids, int32_t batch,
                                             const void* q_host, const void* k_new_host,
                                             const void* v_new_host, const int64_t* slots_host,
                                             float* out_host, pkv_stream_t stream) {
  using namespace pkv;
  if (!g || !pool || !seq_ids || !q_host || !k_new_host || !v_new_host || !slots_host ||
      !out_host || batch <= 0 || batch > g->buckets.back())
    return PKV_ERR_INVALID_ARG;
  const pkv_decode_graph_config& c = g->cfg;
  const int32_t Bmax = g->buckets.back(), mb = c.max_blocks_per_seq;
  int32_t* tables = g->host_meta;
  int32_t* lens = g->host_meta + static_cast<size_t>(Bmax) * mb;
  pkv_status s = seq_batch_tables(pool, seq_ids, batch, mb, tables, lens);
  if (s != PKV_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t qrow = static_cast<size_t>(c.num_q_heads) * c.head_dim * elem_bytes(c.q_dtype);
  const size_t kvrow = static_cast<size_t>(c.num_kv_heads) * c.head_dim * elem_bytes(c.src_dtype);
  const size_t orow = static_cast<size_t>(c.num_q_heads) * c.head_dim * sizeof(float);
  const size_t L = static_cast<size_t>(c.num_layers);
  // Inputs: one staging kernel when every host buffer is mapped page-locked
  // memory, else one copy per buffer.
  const uint8_t* m_tab = mapped(tables);
  const uint8_t* m_q = mapped(q_host);
  const uint8_t* m_k = mapped(k_new_host);
  const uint8_t* m_v = mapped(v_new_host);
  const uint8_t* m_sl = mapped(slots_host);
  if (m_tab && m_q && m_k && m_v && m_sl) {
    StageArgs a{};
    const int64_t tb = static_cast<int64_t>(batch) * mb * 4;
    a.seg[0] = {m_tab, reinterpret_cast<uint8_t*>(c.block_tables), tb, tb, tb, 1};
    const int64_t lb = static_cast<int64_t>(batch) * 4;
    a.seg[1] = {m_tab + static_cast<size_t>(Bmax) * mb * sizeof(int32_t),
                reinterpret_cast<uint8_t*>(c.context_lens), lb, lb, lb, 1};
    const int64_t sb = static_cast<int64_t>(batch) * 8;
    a.seg[2] = {m_sl, reinterpret_cast<uint8_t*>(c.slot_mapping), sb, sb, sb, 1};
    const int64_t qr = static_cast<int64_t>(qrow), kr = static_cast<int64_t>(kvrow);
    const int64_t qb = batch * qr, kb = batch * kr;
    a.seg[3] = {m_q, static_cast<uint8_t*>(c.q), qb, qb, Bmax * qr, static_cast<int32_t>(L)};
    a.seg[4] = {m_k, static_cast<uint8_t*>(c.k_new), kb, kb, Bmax * kr, static_cast<int32_t>(L)};
    a.seg[5] = {m_v, static_cast<uint8_t*>(c.v_new), kb, kb, Bmax * kr, static_cast<int32_t>(L)};
    stage_inputs_kernel<<<dim3(2 * device_sm_count(), kStageSegs), 256, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  } else {
    bool ok =
      cudaMemcpyAsync(c.block_tables, tables, static_cast<size_t>(batch) * mb * sizeof(int32_t),
                      cudaMemcpyHostToDevice, st) == cudaSuccess &&
      cudaMemcpyAsync(c.context_lens, lens, static_cast<size_t>(batch) * sizeof(int32_t),
                      cudaMemcpyHostToDevice, st) == cudaSuccess &&
      cudaMemcpyAsync(c.slot_mapping, slots_host, static_cast<size_t>(batch) * sizeof(int64_t),
                      cudaMemcpyHostToDevice, st) == cudaSuccess &&
      cudaMemcpy2DAsync(c.q, Bmax * qrow, q_host, batch * qrow, batch * qrow, L,
                        cudaMemcpyHostToDevice, st) == cudaSuccess &&
      cudaMemcpy2DAsync(c.k_new, Bmax * kvrow, k_new_host, batch * kvrow, batch * kvrow, L,
                        cudaMemcpyHostToDevice, st) == cudaSuccess &&
      cudaMemcpy2DAsync(c.v_new, Bmax * kvrow, v_new_host, batch * kvrow, batch * kvrow, L,
                        cudaMemcpyHostToDevice, st) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
  }
  s = decode_graph_launch(g, batch, nullptr, stream);
  if (s != PKV_OK) return s;
  if (cudaMemcpy2DAsync(out_host, batch * orow, c.out, Bmax * orow, batch * orow, L,
                        cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

