// mla_decode_paged_static: the dense bf16 decode for callers that cannot
// allocate device memory (for example code running where cudaMalloc is not
// allowed or not wanted: inside another allocator's callback, under a memory
// budget fixed at start-up, or in a plug-in that receives only the tensors).
// It runs exactly the launch sequence of mla_decode_paged, but its scratch
// space is a fixed array compiled into this library instead of a
// caller-provided workspace.
//
// The array is a file-scope __device__ variable, so every GPU on which this
// file's module is loaded holds kStaticScratchBytes of it until the process
// exits (with the default lazy module loading that is each device where this
// entry point has been called; with eager loading, every device).  Host code
// must not pass the array's name to a kernel: on the host it is only a
// stand-in symbol.  Its device address is looked up once per device with
// cudaGetSymbolAddress, on the first call made while that device is current,
// and kept for later calls on that device.  cudaDeviceReset destroys the
// context that address belongs to: the cached address is then stale, so a
// process that resets a device must not call this entry point on it again.
#include <atomic>
#include <cstdio>
#include <mutex>

#include "mla_kernels.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;   // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Per device: the array's device address once looked up (published with release
// order, so a thread that reads it non-null also sees it complete); the lookup
// itself runs under a mutex, so concurrent first calls from several host
// threads look it up once.
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_static_scratch on the current device (looked up once).
int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    p = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
      const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess || !p) {
        std::fprintf(stderr, "mla_decode_paged_static: cudaGetSymbolAddress failed: %s\n",
                     cudaGetErrorString(e));
        return MLA_ERR_CUDA;
      }
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return MLA_OK;
}

}  // namespace

extern "C" {

size_t mla_decode_static_scratch_bytes(void) { return kStaticScratchBytes; }

int mla_decode_paged_static(const mla_dims_t* dims, const mla_opts_t* opts, const void* q,
                            const uint32_t* input_row_offsets, int32_t batch, int32_t total_q,
                            const void* kv_pool, const int32_t* block_table, int32_t block_table_stride,
                            const uint32_t* cache_lens, const void* w_uk, const void* w_uv, void* out,
                            float* lse_out, void* stream) {
  size_t need = 0;
  int st = mla_decode_workspace_size(dims, opts, batch, total_q, &need);
  if (st) return st;
  if (need > kStaticScratchBytes) {
    std::fprintf(stderr,
                 "mla_decode_paged_static: this call needs %zu bytes of scratch, more than the %zu "
                 "compiled in; use fewer query tokens or num_splits, or mla_decode_paged\n",
                 need, kStaticScratchBytes);
    return MLA_ERR_WORKSPACE_TOO_SMALL;
  }
  void* scratch = nullptr;
  if ((st = static_scratch(&scratch))) return st;
  // Nothing in the scratch has to start at zero: the planner rewrites the
  // header and every later kernel writes what it reads within the same call.
  return mla_decode_paged(dims, opts, q, input_row_offsets, batch, total_q, kv_pool, block_table,
                          block_table_stride, cache_lens, w_uk, w_uv, out, lse_out, scratch, kStaticScratchBytes,
                          stream);
}

}  // extern "C"
