// sprint_fc_bwd_static_scratch: the FC backward pass for callers that cannot
// allocate device memory.
//
// sprint_fc_bwd needs caller-provided scratch (the transposed copies its
// weight-gradient GEMM reads). Some callers cannot provide it: code that runs
// under a memory manager which owns every byte of device memory and forbids
// further allocations, or a code path that must not call cudaMalloc/cudaFree
// because those calls may synchronise the device. This entry point takes its
// scratch from a fixed array compiled into the library instead, so it neither
// allocates nor asks the caller to.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its kScratchBytes until the process exits. Host code cannot use
// the array's name as a device pointer, so the first call in each CUDA context
// looks up the array's device address there (cudaGetSymbolAddress, with that
// context's device current) and caches it with the context's unique ID. A
// context created later on the same device (after cudaDeviceReset, say) has a
// new ID and may hold the array at another address, so its first call looks
// the address up again instead of reusing a stale one.
#include <mutex>

#include "common.cuh"

namespace sprint {
namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(24) << 20;  // 24 MiB per device

static __device__ __align__(256) unsigned char g_fc_bwd_scratch[kScratchBytes];

std::mutex g_scratch_mu;
struct ScratchSlot {
    unsigned long long ctx_id;   // unique ID of the context the address belongs to (0: none yet)
    void* addr;
};
ScratchSlot g_scratch[64] = {};

// cuCtxGetCurrent / cuCtxGetId through the runtime's driver entry points (no
// link against libcuda); null if the driver lacks them
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
void ctx_fns(CtxGetCurrentFn* cur, CtxGetIdFn* id) {
    static CtxGetCurrentFn f_cur = nullptr;
    static CtxGetIdFn f_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f_cur = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    *cur = f_cur;
    *id = f_id;
}

// Device address of g_fc_bwd_scratch in the current context (looked up once per context).
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPRINT_ERR_CUDA, "sprint_fc_bwd_static_scratch: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(SPRINT_ERR_UNSUPPORTED, "sprint_fc_bwd_static_scratch: device %d out of range", dev);
    CtxGetCurrentFn get_cur;
    CtxGetIdFn get_id;
    ctx_fns(&get_cur, &get_id);
    if (!get_cur || !get_id)
        return fail(SPRINT_ERR_CUDA, "sprint_fc_bwd_static_scratch: driver lacks cuCtxGetCurrent / cuCtxGetId");
    CUcontext ctx = nullptr;
    if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) {
        // no context current yet: the runtime sets up the device's primary context on this lookup
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fc_bwd_scratch);
        if (e != cudaSuccess || get_cur(&ctx) != CUDA_SUCCESS || !ctx)
            return fail(SPRINT_ERR_CUDA, "sprint_fc_bwd_static_scratch: no CUDA context on device %d", dev);
    }
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS || id == 0)
        return fail(SPRINT_ERR_CUDA, "sprint_fc_bwd_static_scratch: cannot identify the current CUDA context");
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchSlot& slot = g_scratch[dev];
    if (slot.ctx_id != id || !slot.addr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fc_bwd_scratch);
        if (e != cudaSuccess || !p)
            return fail(SPRINT_ERR_CUDA, "sprint_fc_bwd_static_scratch: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        slot.ctx_id = id;
        slot.addr = p;
    }
    *out = slot.addr;
    return SPRINT_OK;
}

}  // namespace
}  // namespace sprint

using namespace sprint;

extern "C" size_t sprint_fc_bwd_static_scratch_bytes(void) { return kScratchBytes; }

extern "C" int sprint_fc_bwd_static_scratch(const float* x, const float* w, const float* wT, const float* dy,
                                            const float* relu_src, float* dx, float* dw, float* db, float alpha,
                                            int accumulate, int N, int in, int out, sprint_stream_t stream) {
    SPRINT_REQUIRE(N >= 1 && in >= 1 && out >= 1, SPRINT_ERR_SHAPE, "%s: need N, in, out >= 1 (got %d, %d, %d)",
                   __func__, N, in, out);
    // the transposed weights are only formed when dx is asked for and wT is absent
    const size_t need = sprint_fc_workspace_size(N, in, out, (wT != nullptr || dx == nullptr) ? 1 : 0);
    SPRINT_REQUIRE(need <= kScratchBytes, SPRINT_ERR_WORKSPACE,
                   "%s: this shape needs %zu bytes of scratch; the library's static scratch holds %zu bytes "
                   "(pass wT, or use sprint_fc_bwd with a caller workspace)",
                   __func__, need, kScratchBytes);
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc) return rc;
    return sprint_fc_bwd(x, w, wT, dy, relu_src, dx, dw, db, alpha, accumulate, N, in, out, scratch, kScratchBytes,
                         stream);
}
