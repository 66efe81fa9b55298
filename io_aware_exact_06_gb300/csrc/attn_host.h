// Host services of the forward's translation unit (attn_fwd.cu) that the
// backward's host code (attn_bwd.cu) shares: one library lock, one error word
// per device, the TMA descriptor encoder.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace attn_host {

// The lock every entry point of the library holds while it touches shared
// host state (devices, workspaces).
std::mutex& lib_mutex();

// Records e as the thread's last CUDA error and returns ATTN_ERR_CUDA.
int lib_cuda_fail(cudaError_t e);

// Device allocations of the library's workspaces, counted for
// attn_device_bytes: every workspace is allocated and released through these.
cudaError_t lib_malloc_raw(void** p, size_t bytes);
void lib_free(void* p);
// Bytes the library holds through lib_malloc (all devices).
size_t lib_device_bytes();
template <class T>
cudaError_t lib_malloc(T** p, size_t bytes) {
  return lib_malloc_raw(reinterpret_cast<void**>(p), bytes);
}

// The current device (checked to be sm_103), its SM count and its error word
// (read by attn_last_device_error).  Call with the lock held.
int lib_device(int* dev, int* sms, int** err);

// 3-D TMA view [tokens, H, d] of a bf16 tensor: box 64 elements x 1 head x
// 128 tokens, 128-byte swizzle.  Call with the lock held.
int lib_make_map(CUtensorMap* map, const void* ptr, int64_t tokens, int H, int d);

}  // namespace attn_host
