// kvq_noalloc.cu -- kvq_decode_attn_noalloc: the decode entry point for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they decode: an engine whose device memory is fully budgeted
// up front by its own pool, a plugin that runs inside a host framework that
// forbids allocations on its hot path, or a real-time loop where an
// allocation's latency or possible failure is not acceptable.  Those callers
// cannot provide kvq_decode_attn's workspace, so this entry point uses a
// fixed scratch array that lives in the library itself instead.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes.
// Every GPU on which the library is loaded holds it until the process exits.
// All calls share it and it keeps the last call's contents, so calls that
// overlap on the GPU (different streams, or different host threads on the
// same device) race on it: serialise them.  The split counters at its start
// are cleared with cudaMemsetAsync before every call.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the device address is fetched with
// cudaGetSymbolAddress once per device, with that device current, the first
// time this entry point runs on it.  Make that first call before any stream
// capture begins.
#include <mutex>

#include "kvq_internal.cuh"

namespace {

constexpr uint64_t kNoAllocScratchBytes = 8ull << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_for_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kvq_status kvq_decode_attn_noalloc(const kvq_config* cfg, const void* layer_buf, int32_t tokens,
                                              const uint16_t* q, uint16_t* out, float* lse,
                                              kvq_stream_t stream) {
  if (!layer_buf || !q || !out) return KVQ_ERR_INVALID_ARG;
  kvq_layout L;
  kvq_status st = kvq_layout_query(cfg, &L);
  if (st != KVQ_OK) return st;
  int32_t n_split = 0, n_qsplit = 0;
  st = kvq_decode_plan(cfg, tokens, &n_split, &n_qsplit);
  if (st != KVQ_OK) return st;
  // the same scratch layout kvq_decode_attn uses: counters, (m, l), accumulators
  const uint64_t ns = (uint64_t)cfg->batch * cfg->n_kv_heads;
  const uint64_t g = (uint64_t)(cfg->n_q_heads / cfg->n_kv_heads);
  const uint64_t cnt = round_up(ns * 4, 256);
  const uint64_t need = n_split > 1
      ? cnt + round_up(ns * n_split * g * 2 * 4, 256) + ns * n_split * g * kvq::kHeadDim * 4
      : 0;
  if (need > kNoAllocScratchBytes) return KVQ_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return KVQ_ERR_CUDA;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (need > 0 && cudaMemsetAsync(scratch, 0, cnt, cs) != cudaSuccess) return KVQ_ERR_CUDA;
  return kvq_decode_attn(cfg, layer_buf, tokens, q, out, lse, scratch, kNoAllocScratchBytes, stream);
}
