// Decode step for callers that cannot allocate device memory.
//
// tb_block_decode needs a caller-provided workspace (the split-K attention
// partials, the query and attention rows, the residual stream and the SwiGLU
// activations of the step).  Some callers cannot obtain one: code that must
// not call cudaMalloc or a framework allocator on its hot path (cudaMalloc and
// cudaFree can synchronise the device and take unbounded time), plugins whose
// host framework owns every byte of device memory and hands out none, and
// runtimes that have no device allocator at all.  tb_block_decode_noalloc
// runs the same decode step with its workspace in a file-scope device array
// of fixed size, so the call itself allocates nothing.
#include <mutex>

#include "common.cuh"

namespace tb {
namespace {

// Largest workspace the no-allocation decode can use: 64 MiB.  The decode of
// 32 sequences with a 16384-row cache at d = 4096, H = 32, Hkv = 8, f = 14336
// needs about 37 MB.  Every GPU that loads this library holds the array until
// the process exits.
constexpr size_t kStaticScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch on the current device, looked up once per
// device (host code cannot use the symbol itself as a device pointer) and kept
// for the life of the process; a cudaDeviceReset after the first call on a
// device would reload the module and could move the array, so it is not
// supported.
void* scratch_on_current_device(cudaError_t* why) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  *why = cudaGetDevice(&dev);
  if (*why != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *why = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *why = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (*why != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace tb

extern "C" TB_API tb_status tb_block_decode_noalloc(const tb_block_cfg* cfg, const void* packed, const void* x,
                                                    void* y, int32_t y_dtype, const tb_kvcache* kv,
                                                    void* stream) {
  // Bad arguments and empty calls are reported or returned by tb_block_decode
  // itself before it touches a workspace.
  const size_t need = (cfg && kv) ? tb_workspace_bytes(cfg, kv->B, kv->T_max, 1) : 0;
  if (need == 0 || kv->B == 0) return tb_block_decode(cfg, packed, x, y, y_dtype, kv, nullptr, 0, stream);
  if (need > tb::kStaticScratchBytes)
    return tb::report(TB_ERR_INVALID_ARG,
                      "tb_block_decode_noalloc: this step needs %zu bytes of workspace, more than the %zu-byte "
                      "static scratch (use tb_block_decode with a caller workspace)",
                      need, tb::kStaticScratchBytes);
  cudaError_t why = cudaSuccess;
  void* ws = tb::scratch_on_current_device(&why);
  if (!ws)
    return tb::report(TB_ERR_CUDA, "tb_block_decode_noalloc: cudaGetSymbolAddress of the static scratch: %s",
                      cudaGetErrorString(why));
  return tb_block_decode(cfg, packed, x, y, y_dtype, kv, ws, tb::kStaticScratchBytes, stream);
}
