// GradBuf accumulation (Algorithm 1, ComputeUpdateVal + UpdateGradient) and
// the parameter-server apply over k pending gradient buffers (Algorithm 2,
// SumGradient + UpdateWeights; DistBelief w' := w - eta*dw with momentum or
// per-parameter Adagrad).
//
// Both are pure streams over HBM: each element is read once from every input
// and written once, with 128-bit loads/stores, streaming cache hints (the
// vectors are far larger than L2), and a grid of a few CTAs per SM looping
// over the vector so that enough bytes are in flight to cover HBM latency.
#include "common.cuh"

namespace sprint {
namespace {

constexpr int kMaxBufs = 16;
constexpr int kThreads = 256;

struct BufPtrs {
    const float* p[kMaxBufs];
};

enum class Opt { SGD, Momentum, Adagrad };

__device__ __forceinline__ float4 ld_stream(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_stream(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

template <Opt OPT>
__device__ __forceinline__ void apply1(float s, float w, float* state, float eta, float hp, float& w_new) {
    if constexpr (OPT == Opt::SGD) {
        w_new = w - eta * s;
    } else if constexpr (OPT == Opt::Momentum) {
        float v = hp * (*state) - eta * s;   // v' = nu*v - eta*S
        *state = v;
        w_new = w + v;                       // W' = W + v'
    } else {
        float g = *state + s * s;            // G' = G + S*S
        *state = g;
        w_new = w - eta * s / (sqrtf(g) + hp);  // W' = W - eta*S/(sqrt(G') + eps)
    }
}

// k is a compile-time constant so the buffer loop unrolls and all k loads of
// one float4 are in flight together.
template <Opt OPT, int K>
__global__ void __launch_bounds__(kThreads) update_kernel(const float* w_in, float* w_out, float* state, BufPtrs bufs,
                                                          size_t n, float eta, float hp) {
    const size_t n4 = n / 4;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 g[K];
#pragma unroll
        for (int j = 0; j < K; ++j) g[j] = ld_stream(bufs.p[j] + 4 * i);
        float4 w = ld_stream(w_in + 4 * i);
        float4 st = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (OPT != Opt::SGD) st = ld_stream(state + 4 * i);
        float4 s = g[0];
#pragma unroll
        for (int j = 1; j < K; ++j) {  // SendBuf = sum_t GradBuf_t, in buffer order
            s.x += g[j].x;
            s.y += g[j].y;
            s.z += g[j].z;
            s.w += g[j].w;
        }
        float4 o;
        apply1<OPT>(s.x, w.x, &st.x, eta, hp, o.x);
        apply1<OPT>(s.y, w.y, &st.y, eta, hp, o.y);
        apply1<OPT>(s.z, w.z, &st.z, eta, hp, o.z);
        apply1<OPT>(s.w, w.w, &st.w, eta, hp, o.w);
        if constexpr (OPT != Opt::SGD) st_stream(state + 4 * i, st);
        st_stream(w_out + 4 * i, o);
    }
    // scalar tail (n % 4 elements), handled by the first CTA
    if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
        const size_t i = 4 * n4 + threadIdx.x;
        float s = bufs.p[0][i];
        for (int j = 1; j < K; ++j) s += bufs.p[j][i];
        float st = (OPT != Opt::SGD) ? state[i] : 0.f;
        float o;
        apply1<OPT>(s, w_in[i], &st, eta, hp, o);
        if constexpr (OPT != Opt::SGD) state[i] = st;
        w_out[i] = o;
    }
}

__global__ void __launch_bounds__(kThreads) gradbuf_kernel(float* buf, const float* grad, size_t n, float alpha,
                                                           int first) {
    const size_t n4 = n / 4;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 g = ld_stream(grad + 4 * i);
        float4 b = first ? make_float4(0.f, 0.f, 0.f, 0.f) : ld_stream(buf + 4 * i);
        b.x += alpha * g.x;
        b.y += alpha * g.y;
        b.z += alpha * g.z;
        b.w += alpha * g.w;
        st_stream(buf + 4 * i, b);
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
        const size_t i = 4 * n4 + threadIdx.x;
        buf[i] = (first ? 0.f : buf[i]) + alpha * grad[i];
    }
}

int stream_grid(size_t n) {
    const size_t n4 = n / 4 + 1;
    size_t want = (n4 + kThreads - 1) / kThreads;
    size_t cap = static_cast<size_t>(num_sms()) * 8;  // 8 x 256 threads per SM
    return static_cast<int>(want < cap ? want : cap);
}

template <Opt OPT>
int launch_update(const char* fn, const float* w_in, float* w_out, float* state, const float* const* bufs, int k,
                  size_t n, float eta, float hp, sprint_stream_t stream) {
    SPRINT_REQUIRE(k >= 1, SPRINT_ERR_SHAPE, "%s: k must be >= 1 (got %d)", fn, k);
    SPRINT_REQUIRE(k <= kMaxBufs, SPRINT_ERR_UNSUPPORTED, "%s: k = %d > %d buffers", fn, k, kMaxBufs);
    if (n == 0) return SPRINT_OK;
    SPRINT_REQUIRE(w_in && w_out && bufs, SPRINT_ERR_INVALID_ARG, "%s: NULL w_in, w_out or bufs", fn);
    SPRINT_REQUIRE(OPT == Opt::SGD || state, SPRINT_ERR_INVALID_ARG, "%s: NULL optimizer state", fn);
    SPRINT_REQUIRE(aligned16(w_in) && aligned16(w_out) && (!state || aligned16(state)), SPRINT_ERR_ALIGN,
                   "%s: w_in, w_out and state must be 16-byte aligned", fn);
    BufPtrs bp{};
    for (int j = 0; j < k; ++j) {
        SPRINT_REQUIRE(bufs[j], SPRINT_ERR_INVALID_ARG, "%s: bufs[%d] is NULL", fn, j);
        SPRINT_REQUIRE(aligned16(bufs[j]), SPRINT_ERR_ALIGN, "%s: bufs[%d] not 16-byte aligned", fn, j);
        bp.p[j] = bufs[j];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int grid = stream_grid(n);
    switch (k) {
#define SPRINT_K(KK) \
    case KK: update_kernel<OPT, KK><<<grid, kThreads, 0, s>>>(w_in, w_out, state, bp, n, eta, hp); break;
        SPRINT_K(1) SPRINT_K(2) SPRINT_K(3) SPRINT_K(4) SPRINT_K(5) SPRINT_K(6) SPRINT_K(7) SPRINT_K(8)
        SPRINT_K(9) SPRINT_K(10) SPRINT_K(11) SPRINT_K(12) SPRINT_K(13) SPRINT_K(14) SPRINT_K(15) SPRINT_K(16)
#undef SPRINT_K
    }
    return check_launch(fn);
}

}  // namespace
}  // namespace sprint

using namespace sprint;

extern "C" int sprint_gradbuf_accumulate(float* buf, const float* grad, size_t n, float alpha, int first,
                                         sprint_stream_t stream) {
    if (n == 0) return SPRINT_OK;
    SPRINT_NONNULL(buf, "buf");
    SPRINT_NONNULL(grad, "grad");
    SPRINT_ALIGNED(buf, "buf");
    SPRINT_ALIGNED(grad, "grad");
    gradbuf_kernel<<<stream_grid(n), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(buf, grad, n, alpha, first);
    return check_launch(__func__);
}

extern "C" int sprint_apply_update_sgd(const float* w_in, float* w_out, const float* const* bufs, int k, size_t n,
                                       float eta, sprint_stream_t stream) {
    return launch_update<Opt::SGD>(__func__, w_in, w_out, nullptr, bufs, k, n, eta, 0.f, stream);
}

extern "C" int sprint_apply_update_momentum(const float* w_in, float* w_out, float* v, const float* const* bufs, int k,
                                            size_t n, float eta, float nu, sprint_stream_t stream) {
    return launch_update<Opt::Momentum>(__func__, w_in, w_out, v, bufs, k, n, eta, nu, stream);
}

extern "C" int sprint_apply_update_adagrad(const float* w_in, float* w_out, float* G, const float* const* bufs, int k,
                                           size_t n, float eta, float eps, sprint_stream_t stream) {
    return launch_update<Opt::Adagrad>(__func__, w_in, w_out, G, bufs, k, n, eta, eps, stream);
}
