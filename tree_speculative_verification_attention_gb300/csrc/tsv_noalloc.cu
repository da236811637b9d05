// tsv_noalloc.cu — greedy tree verification without a caller-provided workspace.
//
// Some callers cannot hand this library a device buffer: code that runs where
// allocation is not allowed or not possible (inside an engine or plugin whose
// allocator owns all device memory, a real-time loop that must never enter the
// CUDA allocator, a host language binding without device-memory management).
// tsv_tree_verify_greedy_noalloc serves them: its scratch (per-request
// completion counters and per-row argmax words) lives in one file-scope
// __device__ array of fixed size, which every GPU that loads the library keeps
// until the process exits.  The caller still passes every input and output.
//
// The array is shared by all calls on a device and keeps the last call's
// contents: the counters and row words, which must start at zero (every call
// leaves them so), are also cleared on the stream at the start of every call.  Calls whose work overlaps on the GPU (different
// streams, no ordering between them) race on the array and give wrong results.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tsv_internal.h"

namespace {

// Fixed scratch: enough for TSV_MAX_BATCH requests of TSV_MAX_NODES rows at any
// vocabulary size (4 bytes per request and 8 per row).
constexpr size_t kNoallocScratchBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device and CUDA
// context.  In host code the symbol itself is only a host-side stand-in for the
// device array, so the kernel must be given the address cudaGetSymbolAddress
// returns.  That address belongs to the context the module was loaded in: after
// cudaDeviceReset (or a release and re-creation of the primary context) the
// module loads again, possibly elsewhere, so the cache keeps the unique id of
// the context it was filled in and looks the address up again when the current
// context's id differs.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Unique id of the calling thread's current context (the driver never reuses
// one within a process).
tsv_status current_context_id(unsigned long long* id) {
  if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || f1 == nullptr ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess || f2 == nullptr)
      return TSV_ERR_CUDA;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return TSV_ERR_CUDA;
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS ? TSV_OK : TSV_ERR_CUDA;
}

// The device address of the scratch array on `device`, which the caller has
// made current (cudaGetDevice), so cudaGetSymbolAddress runs with that device
// current.  Looked up on the first call in each context, then cached.
tsv_status scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return TSV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long id = 0;
  const bool have_ctx = current_context_id(&id) == TSV_OK;
  if (!have_ctx || g_scratch_ptr[device] == nullptr || g_scratch_ctx[device] != id) {
    // cudaGetSymbolAddress also sets up the device's context when no runtime
    // call has yet; its id is read after it.
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      g_scratch_ptr[device] = nullptr;
      return TSV_ERR_CUDA;
    }
    if (current_context_id(&id) != TSV_OK) return TSV_ERR_CUDA;
    g_scratch_ptr[device] = p;
    g_scratch_ctx[device] = id;
  }
  *out = g_scratch_ptr[device];
  return TSV_OK;
}

}  // namespace

extern "C" tsv_status tsv_tree_verify_greedy_noalloc(
    tsv_handle h, const float* logits_d, int64_t V, const int32_t* tree_tokens_d,
    const int32_t* parent_d, const int32_t* node_offsets_d, int32_t B, int32_t N, int32_t* path_d,
    int32_t* accept_len_d, int32_t* bonus_d, int32_t* status_d, void* stream) {
  if (!h) return TSV_ERR_INVALID_ARG;
  size_t need = 0;
  tsv_status st = tsv_tree_verify_greedy_workspace_size(h, B, N, V, &need);
  if (st != TSV_OK) return st;
  if (need > kNoallocScratchBytes) return TSV_ERR_SCRATCH_LIMIT;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return TSV_ERR_CUDA;
  void* scratch = nullptr;
  st = scratch_address(device, &scratch);
  if (st != TSV_OK) return st;
  // The workspace of greedy verification holds B int32 completion counters
  // and N 64-bit row argmax words (tsv_tree_verify_greedy's layout); they
  // must be zero.  Every call leaves them at zero; clearing them here also
  // covers a call that never completed.
  const size_t zeroed_bytes = tsv::greedy_workspace_bytes(B, N);
  if (cudaMemsetAsync(scratch, 0, zeroed_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return TSV_ERR_CUDA;
  return tsv_tree_verify_greedy(h, logits_d, V, tree_tokens_d, parent_d, node_offsets_d, B, N, path_d,
                                accept_len_d, bonus_d, scratch, kNoallocScratchBytes, status_d,
                                stream);
}
