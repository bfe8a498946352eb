// Host-side plumbing of libsprint: thread-local error messages, the device
// status word, and the staleness schedule (host only).
#include <stdarg.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace sprint {

static thread_local char g_err[1024] = "";

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
}

int fail(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return status;
}

static std::atomic<unsigned long long> g_launches{0};

int check_cuda(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPRINT_ERR_CUDA, "%s: CUDA error %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return SPRINT_OK;
}

int check_launch(const char* what, int kernels) {
    g_launches.fetch_add(static_cast<unsigned long long>(kernels), std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPRINT_ERR_CUDA, "%s: CUDA error %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return SPRINT_OK;
}

// The device status word: a file-scope __device__ variable (one per device
// that loads the library); kernels OR flags into it when a bounded wait gives
// up. Host code passes its device address to the kernels.
static __device__ int g_device_status;
static std::mutex g_mu;
static int* g_status[64] = {nullptr};
static int g_sms[64] = {0};

int* device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status[dev] = static_cast<int*>(p);
    }
    return g_status[dev];
}

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!g_sms[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = n > 0 ? n : 148;
    }
    return g_sms[dev];
}

}  // namespace sprint

using namespace sprint;

extern "C" const char* sprint_last_error(void) { return g_err; }

extern "C" int sprint_version(void) { return 100; }

extern "C" uint64_t sprint_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int sprint_device_status(int* flags_out, int reset) {
    SPRINT_NONNULL(flags_out, "flags_out");
    int* p = device_status_ptr();
    if (!p) return fail(SPRINT_ERR_CUDA, "sprint_device_status: no device status word");
    if (cudaDeviceSynchronize() != cudaSuccess) return check_cuda("sprint_device_status");
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return check_cuda("sprint_device_status");
    if (reset && cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return check_cuda("sprint_device_status");
    *flags_out = v;
    if (v) return fail(SPRINT_ERR_DEVICE_FLAG, "a kernel reported a failed bounded wait (flags 0x%x)", v);
    return SPRINT_OK;
}

// One thread waits, with the library's bounded wait, on an mbarrier phase that
// nothing completes (no arrival, no copy, no MMA in flight): the wait gives up
// after limit_ns and sets DEV_FLAG_WAIT_SELFTEST in the status word, and the
// kernel returns. Exercises the failure path every pipelined kernel relies on.
namespace sprint {
__global__ void selftest_wait_kernel(int* status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, status, DEV_FLAG_WAIT_SELFTEST, limit_ns);
    __syncthreads();
}
}  // namespace sprint

extern "C" int sprint_selftest_bounded_wait(uint64_t limit_ns, sprint_stream_t stream) {
    SPRINT_REQUIRE(limit_ns >= 1000 && limit_ns <= 10000000000ull, SPRINT_ERR_INVALID_ARG,
                   "sprint_selftest_bounded_wait: limit_ns must be in [1e3, 1e10] (got %llu)",
                   static_cast<unsigned long long>(limit_ns));
    int* st = device_status_ptr();
    SPRINT_REQUIRE(st != nullptr, SPRINT_ERR_CUDA, "sprint_selftest_bounded_wait: no device status word");
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st, static_cast<unsigned long long>(limit_ns));
    return check_launch("selftest_wait_kernel");
}

// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): the state advances by the
// golden-ratio gamma, and each output is the state passed through the mix.
static inline uint64_t splitmix64_output(uint64_t seed, uint64_t index) {
    uint64_t z = seed + (index + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

extern "C" int sprint_staleness_schedule(uint64_t seed, int steps, int replicas, int max_delay, int32_t* out) {
    SPRINT_REQUIRE(steps >= 0 && replicas >= 1 && max_delay >= 0, SPRINT_ERR_SHAPE,
                   "sprint_staleness_schedule: need steps >= 0, replicas >= 1, max_delay >= 0 (got %d, %d, %d)", steps,
                   replicas, max_delay);
    SPRINT_REQUIRE((long long)steps * replicas < (1ll << 31), SPRINT_ERR_SHAPE,
                   "sprint_staleness_schedule: steps*replicas too large");
    if (steps == 0) return SPRINT_OK;
    SPRINT_NONNULL(out, "out");
    for (long long i = 0; i < (long long)steps * replicas; ++i) {
        uint64_t z = splitmix64_output(seed, (uint64_t)i);
        out[i] = (int32_t)(((z >> 32) * (uint64_t)(max_delay + 1)) >> 32);
    }
    return SPRINT_OK;
}
