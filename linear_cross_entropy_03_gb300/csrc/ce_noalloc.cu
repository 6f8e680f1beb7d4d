// ce_fwd_bwd_noalloc: cross entropy on logits for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace of
// their own: a plugin whose enqueue path is forbidden to allocate, a process
// whose device memory is owned and accounted by another allocator, or a
// latency-critical loop where cudaMalloc's implicit synchronisation and
// unpredictable cost are not acceptable.  This entry point runs the same
// kernels as ce_fwd_bwd, but its scratch (a small header and one fp32 loss
// per row) lives in a file-scope device array that every GPU loading the
// library holds until the process exits.  The caller passes only inputs and
// outputs.
//
// The array is found with cudaGetSymbolAddress once per device context, by
// the first call made with that device current (again after a
// cudaDeviceReset, whose new context holds the array at a new address).
// Every call shares the array: calls that overlap on the GPU (different
// streams without ordering) race on it.
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "flce_internal.h"

namespace flce {
int64_t ce_cta_capacity(int dtype, bool vector_path);
int64_t ce_vector_elems(int dtype, bool vector_path);
}  // namespace flce

namespace {

constexpr size_t kHeaderBytes = 256;  // WorkspaceHeader, rounded up
constexpr size_t kArrivalWordOffset = 192;  // the single-launch form's tagged arrival counter
static_assert(sizeof(flce::WorkspaceHeader) <= kArrivalWordOffset, "header overlaps the arrival word");
constexpr size_t kScratchBytes = kHeaderBytes + sizeof(float) * FLCE_NOALLOC_MAX_ROWS;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
struct ScratchSlot {
  unsigned long long ctx_id;  // context the address belongs to (0: none yet)
  void* addr;
};
ScratchSlot g_scratch[64] = {};

// Unique id of the calling thread's current context (0 if unavailable), from
// the driver entry points the runtime hands out.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the array in the current device's context (host code
// cannot use the symbol itself as an address): looked up the first time a
// context is seen, then reused while that context lives.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchSlot& slot = g_scratch[dev];
  const unsigned long long ctx = current_context_id();  // 0 before the runtime set up this thread's context
  if (ctx != 0 && slot.ctx_id == ctx && slot.addr != nullptr) return slot.addr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
  slot.addr = p;
  slot.ctx_id = current_context_id();  // the lookup has made the device's context current
  return slot.addr;
}

bool aligned_to(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// A 40-bit tag no earlier call of this process gave the shared array's
// counters.
unsigned long long next_nonce() {
  static std::atomic<unsigned long long> nonce{0x7F4A7C159E3779B9ull};
  return (nonce.fetch_add(1, std::memory_order_relaxed) + 1) & ((1ull << 40) - 1);
}
int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

using namespace flce;

extern "C" flce_status_t ce_fwd_bwd_noalloc(const void* logits, int dtype, void* grad_logits,
                                            const int64_t* target, int64_t N, int64_t V,
                                            int64_t ignore_index, int reduction, float grad_scale,
                                            const float* grad_out_none, float* loss,
                                            int32_t* status_dev, flce_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (dtype != FLCE_DTYPE_BF16 && dtype != FLCE_DTYPE_FP32 && dtype != FLCE_DTYPE_FP16) return FLCE_ERR_UNSUPPORTED;
  if (N < 0 || V < 1 || reduction < 0 || reduction > 2) return FLCE_ERR_INVALID_ARG;
  if (N > FLCE_NOALLOC_MAX_ROWS) return FLCE_ERR_UNSUPPORTED;  // beyond the static scratch
  if (loss == nullptr || (N > 0 && (logits == nullptr || target == nullptr))) return FLCE_ERR_INVALID_ARG;
  if (grad_out_none != nullptr && reduction != FLCE_REDUCTION_NONE) return FLCE_ERR_INVALID_ARG;
  const size_t esz = dtype == FLCE_DTYPE_FP32 ? 4 : 2;
  if (!aligned_to(logits, esz) || !aligned_to(grad_logits, esz) || !aligned_to(target, 8) ||
      !aligned_to(loss, 4))
    return FLCE_ERR_MISALIGNED;
  if (grad_logits != nullptr && grad_logits != logits) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(logits), b = reinterpret_cast<uintptr_t>(grad_logits);
    const uintptr_t bytes = static_cast<uintptr_t>(N) * V * esz;
    if (a < b + bytes && b < a + bytes) return FLCE_ERR_INVALID_ARG;
  }
  uint8_t* scratch = static_cast<uint8_t*>(scratch_address());
  if (scratch == nullptr) return FLCE_ERR_CUDA;

  WorkspaceHeader* hdr = reinterpret_cast<WorkspaceHeader*>(scratch);
  int* status = status_dev != nullptr ? status_dev : &hdr->status;
  float* loss_rows =
      reduction == FLCE_REDUCTION_NONE ? loss : reinterpret_cast<float*>(scratch + kHeaderBytes);

  const bool ptrs16 = aligned_to(logits, 16) && (grad_logits == nullptr || aligned_to(grad_logits, 16));
  const bool vec = (static_cast<size_t>(V) * esz) % 16 == 0 && ptrs16;
  if (N > 0 && N <= kCeSelfCountMaxRows && ce_rows_single_launch_ok(V, dtype, vec, ptrs16)) {
    // one launch: the row kernel counts the targets itself and finds the CTA
    // that adds the loss partials by a nonce-tagged counter in the scratch
    // header, so nothing needs zeroing first
    CeParams p = {};
    p.logits = logits;
    p.grad = grad_logits;
    p.target = target;
    p.N = N;
    p.V = V;
    p.ignore_index = ignore_index;
    p.reduction = reduction;
    p.grad_scale = grad_scale;
    p.grad_out = grad_out_none;
    p.loss_rows = loss_rows;
    p.status = status_dev;
    p.cluster = 1;
    p.seg_len = V;
    p.loss_out = reduction != FLCE_REDUCTION_NONE ? loss : nullptr;
    p.self_count = 1;
    p.done_flags = reinterpret_cast<unsigned long long*>(scratch + kArrivalWordOffset);
    p.nonce = next_nonce();
    return launch_ce_rows(p, dtype, vec, ptrs16, false, stream) == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA;
  }

  // The header (valid-target count, block ticket, status) must start at zero.
  if (cudaMemsetAsync(hdr, 0, kHeaderBytes, stream) != cudaSuccess) return FLCE_ERR_CUDA;
  if (launch_count_targets(target, N, V, ignore_index, hdr, 0, 0, status, nullptr, nullptr, 0, nullptr, stream) !=
      cudaSuccess)
    return FLCE_ERR_CUDA;
  if (N > 0) {
    const int64_t cap = ce_cta_capacity(dtype, vec);
    const int64_t epv = ce_vector_elems(dtype, vec);
    int64_t cl = ceil_div64(V, cap);
    cl = cl > 8 ? 8 : (cl < 1 ? 1 : cl);
    int64_t seg = ceil_div64(ceil_div64(V, cl), epv) * epv;
    cl = ceil_div64(V, seg);
    CeParams p = {};
    p.logits = logits;
    p.grad = grad_logits;
    p.target = target;
    p.N = N;
    p.V = V;
    p.ignore_index = ignore_index;
    p.reduction = reduction;
    p.grad_scale = grad_scale;
    p.grad_out = grad_out_none;
    p.loss_rows = loss_rows;
    p.n_valid = &hdr->n_valid;
    p.status = status;
    p.cluster = static_cast<int>(cl);
    p.seg_len = seg;
    if (launch_ce_rows(p, dtype, vec, ptrs16, true, stream) != cudaSuccess) return FLCE_ERR_CUDA;
  }
  if (reduction != FLCE_REDUCTION_NONE &&
      launch_loss_reduce(loss_rows, N, reduction, &hdr->n_valid, loss, stream, N > 0) != cudaSuccess)
    return FLCE_ERR_CUDA;
  return FLCE_OK;
}
