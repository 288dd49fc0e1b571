// moe_dispatch_align_noalloc: the capacity dispatch and padded-block alignment
// of moe_dispatch_align, for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: a serving loop whose
// device memory is fixed once at start-up, or code running inside another
// framework that owns the allocator and forbids new allocations while it
// runs.  This entry point allocates nothing.  Its scratch (per-route ranks,
// per-tile expert counts, segment offsets and a status word) lives in one
// file-scope device array of fixed size, which every GPU that loads this
// library holds until the process exits.
//
// Host code never uses the array's name as an address: on the host that name
// is only a stand-in for the device symbol.  The device address is obtained
// with cudaGetSymbolAddress once per device context, with that device
// current, on the first call made in it, and passed to the kernels.  A new
// context on the device (after cudaDeviceReset, say) reloads the module and
// moves the array, so the address is looked up again whenever the current
// context's unique id differs from the one it was found in.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "moe_api.h"

namespace {

// Largest batch this entry point accepts: T*k routes.
constexpr int64_t kMaxRoutes = 65536;
constexpr int kMaxExperts = 256;
constexpr int kMaxCountTiles = (int)(kMaxRoutes / moe::kDispatchTile);

// Word offsets inside the scratch array.
constexpr size_t kStatusWord = 0;                  // word 0; words 1..63 pad to 256 bytes
constexpr size_t kRankOff = 64;                    // rank of each route inside its 1024-route tile
constexpr size_t kTileCountOff = kRankOff + kMaxRoutes;                        // [tiles][N]
constexpr size_t kSegOffOff = kTileCountOff + (size_t)kMaxCountTiles * kMaxExperts;  // [N]
constexpr size_t kScratchWords = kSegOffOff + kMaxExperts;                      // 82,240 words, ~321 KB

static __device__ __align__(256) int32_t g_dispatch_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  int32_t* addr = nullptr;
  unsigned long long ctx_id = 0;   // unique id of the context the address belongs to
};
ScratchAddr g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Unique id of the calling thread's current context (0 if none).  The
// driver entry points are looked up through the runtime, as for the tensor
// maps, so the library needs no link against the driver library.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array on the current device, looked up with
// that device current, again whenever the device's context has changed.
moe_status scratch_on_current_device(int32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  unsigned long long ctx_id = 0;
  const bool have_ctx = current_context_id(&ctx_id);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& a = g_scratch_addr[dev];
  if (!have_ctx || !a.addr || a.ctx_id != ctx_id) {
    // (this runtime call also makes the device's context current if no
    // runtime call has done so on this thread yet)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    if (!current_context_id(&ctx_id)) return MOE_ERR_CUDA;
    a.addr = static_cast<int32_t*>(p);
    a.ctx_id = ctx_id;
  }
  *out = a.addr;
  return MOE_OK;
}

bool ok_ptr(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_dispatch_align_noalloc(const moe_config* cfg, int32_t T,
                                                 const int32_t* topk_idx, uint8_t* route_kept,
                                                 int32_t* route_pos, int32_t* sorted_route_ids,
                                                 int32_t* block_expert, int32_t* num_padded,
                                                 int32_t* expert_counts, int32_t* num_dropped,
                                                 int32_t* status_out, void* stream) {
  const moe_status cs = moe_check_config(cfg);
  if (cs != MOE_OK) return cs;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  // the drop policy only, as moe_dispatch_align
  if (cfg->routing != MOE_ROUTING_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;
  if (cfg->overflow_policy == MOE_OVERFLOW_REROUTE && moe_capacity(cfg, T) >= 0) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * cfg->top_k > kMaxRoutes) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch
  if (T == 0) return MOE_OK;
  if (!ok_ptr(topk_idx) || !ok_ptr(route_kept) || !ok_ptr(route_pos) || !ok_ptr(sorted_route_ids) ||
      !ok_ptr(block_expert) || !ok_ptr(num_padded) || !ok_ptr(expert_counts) || !ok_ptr(num_dropped) ||
      (status_out && (reinterpret_cast<uintptr_t>(status_out) & 3u)))
    return MOE_ERR_INVALID_ARG;
  int32_t* scratch = nullptr;
  const moe_status ss = scratch_on_current_device(&scratch);
  if (ss != MOE_OK) return ss;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the status word must start
  // at zero; ranks, tile counts and offsets are fully rewritten before use.
  if (cudaMemsetAsync(scratch + kStatusWord, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  moe::launch_dispatch(topk_idx, T, cfg->num_experts, cfg->top_k, cfg->block_size, moe_capacity(cfg, T),
                       route_kept, route_pos, sorted_route_ids, block_expert, num_padded, expert_counts,
                       num_dropped, scratch + kRankOff, scratch + kTileCountOff, scratch + kSegOffOff,
                       scratch + kStatusWord, s);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  if (status_out && cudaMemcpyAsync(status_out, scratch + kStatusWord, sizeof(int32_t),
                                    cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
