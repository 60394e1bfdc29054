// paged_gqa_decode_noalloc: the decode call for callers that cannot allocate
// device memory.
//
// Some callers have no way to call cudaMalloc: a plug-in running inside a host
// program that owns the whole device-memory budget, or a serving loop that
// must not allocate once it has started.  Such a caller passes only its
// inputs and outputs; the split-K workspace comes from the file-scope array
// below, which every GPU that loads this library keeps until the process
// exits.  It is shared by every call on a device, so calls whose kernels may
// overlap on the GPU race on it.
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>
#include <stdio.h>

#include "internal.h"
#include "pkv.h"

namespace pkv {

// Workspace of the allocation-free entry point (see PKV_NOALLOC_WORKSPACE_BYTES).
static __device__ __align__(256) uint8_t g_noalloc_workspace[PKV_NOALLOC_WORKSPACE_BYTES];

// Device address of g_noalloc_workspace on `device`, which is current.  Host
// code must not use the symbol itself: on the host it names a stand-in, not
// device memory.  Outside stream capture the address is looked up on every
// call (a host-side lookup, no stream work), so a device reset that reloads
// the library's module cannot leave a stale address behind; while `stream`
// is being captured the address from the last uncaptured call on the device
// is used, and a first call under capture is refused.
static int noalloc_workspace_address(int device, bool capturing, uint8_t** out) {
  static std::mutex mu;
  static uint8_t* addr[64] = {nullptr};
  if (device < 0 || device >= 64) {
    set_last_error("paged_gqa_decode_noalloc", "device index out of range");
    return PKV_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (capturing) {
    if (addr[device] == nullptr) {
      set_last_error("paged_gqa_decode_noalloc",
                     "first call on this device made during stream capture; call it once before capturing");
      return PKV_ERR_CUDA;
    }
  } else {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
    if (e != cudaSuccess) return cuda_status(e, "cudaGetSymbolAddress(noalloc workspace)");
    addr[device] = static_cast<uint8_t*>(p);
  }
  *out = addr[device];
  return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" int paged_gqa_decode_noalloc(const void* q, const void* kv_pool, int num_pages,
                                        const int32_t* block_tables, int bt_row_stride,
                                        int max_blocks, const int32_t* seq_lens, int num_seqs,
                                        int max_seq_len, void* out, float scale, int* d_err,
                                        void* stream) {
  // every check that needs no device comes first: a rejected call touches
  // neither the GPU nor the shared array
  int rc = decode_check_args(q, kv_pool, num_pages, block_tables, bt_row_stride, max_blocks,
                             seq_lens, num_seqs, out, scale);
  if (rc != PKV_OK || num_seqs == 0) return rc;
  bool capturing = false;
  if (stream != nullptr) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap);
    if (e != cudaSuccess) return cuda_status(e, "cudaStreamIsCapturing");
    capturing = cap != cudaStreamCaptureStatusNone;
  }
  int dev = 0;
  rc = bind_stream_device(stream, &dev);
  if (rc != PKV_OK) return rc;
  const size_t need = paged_gqa_decode_workspace_bytes(num_seqs);
  if (need == 0) {
    set_last_error("paged_gqa_decode_noalloc", "cannot size the workspace on this device");
    return PKV_ERR_CUDA;
  }
  if (need > (size_t)PKV_NOALLOC_WORKSPACE_BYTES) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "%d sequences need %zu workspace bytes; the static workspace holds %d",
             num_seqs, need, (int)PKV_NOALLOC_WORKSPACE_BYTES);
    set_last_error("paged_gqa_decode_noalloc", msg);
    return PKV_ERR_WORKSPACE_TOO_SMALL;
  }
  uint8_t* ws = nullptr;
  rc = noalloc_workspace_address(dev, capturing, &ws);
  if (rc != PKV_OK) return rc;
  // The per-segment arrival counters at the front of the workspace must be
  // zero when a call starts; clear them on the caller's stream every time.
  const size_t counters = (size_t)8 * num_seqs * sizeof(uint32_t);
  cudaError_t e = cudaMemsetAsync(ws, 0, counters, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e, "cudaMemsetAsync(noalloc counters)");
  return paged_gqa_decode(q, kv_pool, num_pages, block_tables, bt_row_stride, max_blocks,
                          seq_lens, num_seqs, max_seq_len, out, scale, ws,
                          (size_t)PKV_NOALLOC_WORKSPACE_BYTES, d_err, stream);
}
