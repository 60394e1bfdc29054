// C-ABI utilities: status strings, RoPE tables (host set-up), the device
// error word reader, and device/stream binding.
//
// This file is compiled with -ffp-contract=off: the RoPE frequency and table
// arithmetic must round exactly as written (no fused multiply-add), so the
// tables are reproducible across x86-64 and AArch64 hosts.
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>
#include <stdint.h>
#include <stdio.h>

#include "internal.h"
#include "pkv.h"

namespace pkv {

static thread_local char g_last_error[256] = "";

void set_last_error(const char* where, const char* what) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where ? where : "?", what ? what : "?");
}

int bind_stream_device(void* stream, int* device_out) {
  int dev = 0;
  cudaError_t e;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (stream != nullptr) {
    e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap);
    if (e != cudaSuccess) return cuda_status(e, "cudaStreamIsCapturing");
  }
  if (stream != nullptr && cap == cudaStreamCaptureStatusNone) {
    e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &dev);
    if (e != cudaSuccess) return cuda_status(e, "cudaStreamGetDevice");
    int cur = -1;
    e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
    if (cur != dev) {
      e = cudaSetDevice(dev);
      if (e != cudaSuccess) return cuda_status(e, "cudaSetDevice");
    }
  } else {
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
  }
  *device_out = dev;
  return PKV_OK;
}

int sm_count(int device) {
  static std::mutex mu;
  static int cache[64] = {0};
  if (device < 0 || device >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      (void)cudaGetLastError();
      return 0;
    }
    cache[device] = n;
  }
  return cache[device];
}

}  // namespace pkv

using namespace pkv;

extern "C" const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARGUMENT: return "PKV_ERR_INVALID_ARGUMENT";
    case PKV_ERR_MISALIGNED: return "PKV_ERR_MISALIGNED";
    case PKV_ERR_UNSUPPORTED_SHAPE: return "PKV_ERR_UNSUPPORTED_SHAPE";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "PKV_ERR_WORKSPACE_TOO_SMALL";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_DEVICE_INDEX: return "PKV_ERR_DEVICE_INDEX";
    case PKV_ERR_POOL_EXHAUSTED: return "PKV_ERR_POOL_EXHAUSTED";
    case PKV_ERR_REQUEST_TOO_LARGE: return "PKV_ERR_REQUEST_TOO_LARGE";
    case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT";
    default: return "PKV_ERR_UNKNOWN";
  }
}

extern "C" const char* pkv_last_error(void) { return g_last_error; }

extern "C" int pkv_version(void) { return 10000 * 0 + 100 * 2 + 0; }

extern "C" int pkv_rope_inv_freq_plain(double* inv_freq, double theta) {
  if (!inv_freq || !(theta > 1.0)) return PKV_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < PKV_ROPE_PAIRS; ++i)
    inv_freq[i] = pow(theta, -(2.0 * (double)i) / (double)PKV_HEAD_DIM);
  return PKV_OK;
}

extern "C" int pkv_rope_inv_freq_llama3(double* inv_freq, double theta, double factor,
                                        double low_freq_factor, double high_freq_factor,
                                        int original_max_pos) {
  if (!inv_freq || !(factor > 0.0) || !(high_freq_factor > low_freq_factor) ||
      !(low_freq_factor > 0.0) || original_max_pos < 1)
    return PKV_ERR_INVALID_ARGUMENT;
  int rc = pkv_rope_inv_freq_plain(inv_freq, theta);
  if (rc != PKV_OK) return rc;
  const double orig = (double)original_max_pos;
  const double low_wavelen = orig / low_freq_factor;
  const double high_wavelen = orig / high_freq_factor;
  const double two_pi = 6.283185307179586;  // 2 * pi rounded to double
  for (int i = 0; i < PKV_ROPE_PAIRS; ++i) {
    const double f = inv_freq[i];
    const double wavelen = two_pi / f;
    if (wavelen < high_wavelen) {
      inv_freq[i] = f;
    } else if (wavelen > low_wavelen) {
      inv_freq[i] = f / factor;
    } else {
      const double smooth = (orig / wavelen - low_freq_factor) / (high_freq_factor - low_freq_factor);
      inv_freq[i] = (1.0 - smooth) * f / factor + smooth * f;
    }
  }
  return PKV_OK;
}

extern "C" int pkv_rope_table_fill(float* host_cos, float* host_sin, int max_pos,
                                   const double* inv_freq) {
  if (!host_cos || !host_sin || !inv_freq || max_pos < 1) return PKV_ERR_INVALID_ARGUMENT;
  for (int p = 0; p < max_pos; ++p) {
    for (int i = 0; i < PKV_ROPE_PAIRS; ++i) {
      const double ang = (double)p * inv_freq[i];
      host_cos[(size_t)p * PKV_ROPE_PAIRS + i] = (float)cos(ang);
      host_sin[(size_t)p * PKV_ROPE_PAIRS + i] = (float)sin(ang);
    }
  }
  return PKV_OK;
}

extern "C" int pkv_read_device_error(int* d_err, void* stream, int clear, int* code_out) {
  if (!d_err || !code_out) return PKV_ERR_INVALID_ARGUMENT;
  int dev = 0;
  int rc = bind_stream_device(stream, &dev);
  if (rc != PKV_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, d_err, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e, "pkv_read_device_error");
  *code_out = host;
  if (clear) {
    e = cudaMemsetAsync(d_err, 0, sizeof(int), st);
    if (e != cudaSuccess) return cuda_status(e, "pkv_read_device_error clear");
  }
  return PKV_OK;
}
