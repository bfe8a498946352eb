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
// the array's name as a device pointer, so the first call on each device looks
// up its device address (cudaGetSymbolAddress, with that device current) and
// caches it; later calls reuse the cached address.
#include <mutex>

#include "common.cuh"

namespace sprint {
namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(24) << 20;  // 24 MiB per device

static __device__ __align__(256) unsigned char g_fc_bwd_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {nullptr};

// Device address of g_fc_bwd_scratch on the current device (looked up once).
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPRINT_ERR_CUDA, "sprint_fc_bwd_static_scratch: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(SPRINT_ERR_UNSUPPORTED, "sprint_fc_bwd_static_scratch: device %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fc_bwd_scratch);
        if (e != cudaSuccess || !p)
            return fail(SPRINT_ERR_CUDA, "sprint_fc_bwd_static_scratch: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
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
