// tp_row_linear_reduce_noalloc: the fused row-parallel linear + rank-ordered
// reduction without any device allocation by the library or the caller.
//
// The regular entry point needs a caller-provided workspace for the GEMM's
// split partials and arrival tickets.  Some callers cannot allocate one: a
// plug-in that a host framework hands only its input and output tensors (the
// framework owns every allocation), or a latency-critical loop that cannot
// afford cudaMalloc's implicit device-wide synchronisation.  This entry point
// keeps that scratch in one fixed array in device memory instead.
#include <cuda_runtime.h>

#include <mutex>

#include "tp.h"

namespace tpk {
bool noalloc_fits(int M, int out_rows, int num_sms, size_t ticket_bytes, size_t partial_bytes,
                  int max_tokens);
tp_status row_reduce_in_scratch(const tp_model* m, int32_t layer, int32_t which, const tp_bf16* x,
                                int64_t x_rank_stride, int64_t ldx, int32_t M,
                                const tp_bf16* residual, tp_bf16* y, void* scratch,
                                size_t ticket_bytes, size_t partial_bytes, int32_t max_tokens,
                                cudaStream_t st);
}  // namespace tpk

namespace {
constexpr int32_t kMaxTokens = 64;                               // decode-sized batches
constexpr size_t kTicketBytes = 16 * 1024;                       // 4096 output tiles
constexpr size_t kPartialBytes = 160ull * 2 * 64 * 128 * 4;      // 160 CTAs x 2 x [64 x 128] fp32
constexpr size_t kScratchBytes = kTicketBytes + kPartialBytes;   // 10 MiB + 16 KiB
}  // namespace

// The scratch itself: every GPU that loads the library holds it until the
// process exits.  In host code this name is only a stand-in for the device
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char tp_noalloc_scratch[kScratchBytes];

namespace {
std::mutex g_mu;
constexpr int kMaxDevices = 256;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, resolved once
// per device (with that device current) and cached for the life of the
// process.  A cudaDeviceReset destroys the context the address belongs to,
// so the entry point must not be called on a device after it was reset.
tp_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, tp_noalloc_scratch) != cudaSuccess || !p) return TP_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return TP_OK;
}
}  // namespace

extern "C" tp_status tp_row_linear_reduce_noalloc(const tp_model* m, int32_t layer, int32_t which,
                                                  const tp_bf16* x, int64_t x_rank_stride,
                                                  int64_t ldx, int32_t M, const tp_bf16* residual,
                                                  tp_bf16* y, void* stream) {
  void* scratch = nullptr;
  tp_status s = scratch_address(&scratch);
  if (s != TP_OK) return s;
  return tpk::row_reduce_in_scratch(m, layer, which, x, x_rank_stride, ldx, M, residual, y, scratch,
                                    kTicketBytes, kPartialBytes, kMaxTokens,
                                    static_cast<cudaStream_t>(stream));
}

extern "C" int32_t tp_row_linear_reduce_noalloc_fits(int32_t M, int32_t hidden, int32_t num_sms) {
  return tpk::noalloc_fits(M, hidden, num_sms, kTicketBytes, kPartialBytes, kMaxTokens) ? 1 : 0;
}
