// pkv_decode_attn_static_scratch: split-KV decode attention plus the merge,
// for callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers: plugin
// interfaces of a host framework that give out no workspace, runtimes whose
// device memory is already reserved by another allocator, or latency-critical
// loops where cudaMalloc's implicit device synchronisation is not acceptable.
// Such a caller has nowhere to put the split partials (o_part / ml_part), so
// this entry point keeps them in one file-scope device array instead.
//
// The array is a static __device__ variable: every GPU that loads libpkv
// holds its kStaticScratchBytes until the process exits.  Host code cannot
// use the array's name as a device address (in host code it names a host-side
// stand-in), so the device address is looked up with cudaGetSymbolAddress
// once per device, with that device current, on the first call made on it.
// That first call therefore does a runtime query and should come before any
// stream capture.  Nothing here calls cudaMalloc, cudaFree or any allocating
// library routine.
//
// Every call shares the one array and leaves its last contents behind.
// Nothing in it needs to start at zero: for every (request, head, split) the
// merge reads, the attention kernel of the same call has written it first.
// Calls whose kernels overlap on the GPU (two streams, or two host threads)
// race on the array and give wrong results; issue them in order.
#include <mutex>

#include "kernels.cuh"

namespace pkv {
namespace {

constexpr size_t kStaticScratchBytes = PKV_STATIC_SCRATCH_BYTES;
static_assert(kStaticScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) float g_static_scratch[kStaticScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
float *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_static_scratch on the current device (looked up once).
cudaError_t scratch_address(float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_decode_attn_static_scratch(const pkv_workspace *ws, int batch,
                                                     int layer, const void *q, float scale,
                                                     int num_splits, int flags,
                                                     pkv_stream_t stream) {
  if (!ws || batch < 0 || num_splits < 1) return PKV_ERR_INVALID;
  // The size check below multiplies these: reject what the shape check of
  // pkv_decode_attn would, before they can make `need` small or negative.
  if (ws->head_dim <= 0 || ws->n_q_heads <= 0) return PKV_ERR_INVALID;
  const long long per_split = (long long)ws->head_dim + 2;  // o row + (m, l)
  const long long need = (long long)batch * ws->n_q_heads * num_splits * per_split * 4;
  if (num_splits > 1 && need > (long long)kStaticScratchBytes) return PKV_ERR_CAPACITY;
  pkv_workspace w = *ws;
  if (num_splits > 1) {
    float *base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return PKV_ERR_CUDA;
    const long long n_o = (long long)batch * ws->n_q_heads * num_splits * ws->head_dim;
    w.o_part = base;
    w.ml_part = base + n_o;  // n_o * 4 bytes is a multiple of 32: ml stays aligned
    // The partial buffers only have to hold this call's [batch, Hq, S, *]
    // block: the array's size, checked above, bounds num_splits here, not
    // the caller's max_splits.
    w.max_splits = num_splits;
    if (w.max_batch < batch) return PKV_ERR_CAPACITY;
  }
  pkv_status st = pkv_decode_attn(&w, batch, layer, q, scale, num_splits, flags, stream);
  if (st != PKV_OK || num_splits == 1) return st;
  return pkv_merge_partials(&w, batch, num_splits, flags, stream);
}
