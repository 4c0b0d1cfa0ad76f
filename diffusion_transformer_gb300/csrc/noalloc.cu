// dit_block_forward_noalloc: the whole-block forward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine): a plugin running inside a host
// application whose allocator owns all device memory, or a latency-bound loop in which an
// allocation's implicit device synchronisation is not allowed. They can still pass their inputs and
// outputs. This entry point gives them the block forward with its scratch (the norm outputs, q, k,
// transposed v, the attention output and the SwiGLU output) in a file-scope static device array of
// kStaticScratchBytes. Every GPU that loads the library holds that array until the process exits.
//
// Set-up: the first call on a device, with that device current, looks up the array's device address
// with cudaGetSymbolAddress (host code cannot use the symbol itself: in host code it names a
// host-side stand-in, not device memory). That first call should come before any stream capture.
//
// Every call shares the one array and it keeps the previous call's contents. Nothing in it has to
// start at zero: each call writes every scratch byte its kernels read before reading it (rows beyond
// the sequence are never read from memory; the tile loads fill them with zeros). Calls whose work
// overlaps on the GPU (different streams, or different host threads) race on the array.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "../../include/dit.h"
#include "internal.h"

namespace {

// 64 MiB: enough for the 512x512-image block (hidden 3072, ffn 12288, 1088 rows needs 60.2 MB).
constexpr size_t kStaticScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_block_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the static scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DIT_ECUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_block_scratch) != cudaSuccess || p == nullptr) return DIT_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DIT_OK;
}

}  // namespace

extern "C" {

size_t dit_block_noalloc_max_bytes(void) { return kStaticScratchBytes; }

int dit_block_forward_noalloc(const dit_dims* dims, const dit_block_w* w, float* txt, int L, float* img, int N,
                              const float* txt_cos, const float* txt_sin, const float* img_cos, const float* img_sin,
                              const dit_mod* mod, dit_stream_t stream) {
  // every argument check comes before the first CUDA call, as in the other entry points
  int rc = dit::check_block_call_without_workspace(dims, w, txt, L, img, N, txt_cos, txt_sin, img_cos, img_sin, mod);
  if (rc != DIT_OK) return rc;
  const size_t need = dit_workspace_bytes(dims, L, N, 0);
  if (need == 0) return DIT_EINVAL;
  if (need > kStaticScratchBytes) return DIT_EWORKSPACE;  // the shape needs more than the static array
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != DIT_OK) return rc;
  return dit_block_forward(dims, w, txt, L, img, N, txt_cos, txt_sin, img_cos, img_sin, mod, scratch,
                           kStaticScratchBytes, stream);
}

}  // extern "C"
