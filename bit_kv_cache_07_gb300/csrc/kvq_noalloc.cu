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
// cudaGetSymbolAddress, with the device current: on the first call on a
// device, and again on every call whose stream is not being captured (after
// a cudaDeviceReset the library's module is loaded anew and the array may sit
// elsewhere).  A call made during stream capture reuses the address of the
// last call outside capture, so make one call on each device before any
// stream capture begins (and again after a device reset).
#include <mutex>

#include "kvq_internal.cuh"

namespace {

constexpr uint64_t kNoAllocScratchBytes = 8ull << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// Device address of the scratch array on the current device: looked up
// whenever `st` is not capturing, remembered for calls made during capture.
cudaError_t scratch_for_current_device(cudaStream_t st, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (cap == cudaStreamCaptureStatusNone || !g_scratch_ptr[dev]) {
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
  kvq::DecodeParams p;
  bool persistent = false;
  uint64_t layout_ws = 0;
  kvq_status st = kvq::decode_setup(cfg, layer_buf, tokens, q, out, lse, &p, &persistent, &layout_ws);
  if (st != KVQ_OK) return st;
  // the split plan widened to this device's SMs, as kvq_decode_attn uses it,
  // when its partials fit the scratch; else the narrower host plan
  kvq::DecodeParams host_plan = p;
  uint64_t need = 0;
  st = kvq::decode_plan_device(&p, persistent, &need, /*widen=*/true);
  if (st != KVQ_OK) return st;
  if (need > kNoAllocScratchBytes) {
    p = host_plan;
    st = kvq::decode_plan_device(&p, persistent, &need, /*widen=*/false);
    if (st != KVQ_OK) return st;
  }
  if (need > kNoAllocScratchBytes) return KVQ_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  if (scratch_for_current_device(cs, &scratch) != cudaSuccess) return KVQ_ERR_CUDA;
  // the split counters sit at the start of the scratch and must start at zero
  const uint64_t cnt = round_up((uint64_t)cfg->batch * cfg->n_kv_heads * 4, 256);
  if (need > 0 && cudaMemsetAsync(scratch, 0, cnt, cs) != cudaSuccess) return KVQ_ERR_CUDA;
  return kvq::decode_launch(&p, persistent, scratch, cs);
}
