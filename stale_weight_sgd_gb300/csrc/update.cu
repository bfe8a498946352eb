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

__device__ __forceinline__ float4 ld_stream(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_stream(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

// k is a compile-time constant so the buffer loop unrolls and all k loads of
// one float4 are in flight together.
template <int OPT, int K>
__global__ void __launch_bounds__(kThreads) update_kernel(const float* w_in, float* w_out, float* state, BufPtrs bufs,
                                                          size_t n, float eta, float hp, float wd) {
    const size_t n4 = n / 4;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 g[K];
#pragma unroll
        for (int j = 0; j < K; ++j) g[j] = ld_stream(bufs.p[j] + 4 * i);
        float4 w = ld_stream(w_in + 4 * i);
        float4 st = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (OPT != PS_SGD) st = ld_stream(state + 4 * i);
        float4 s = g[0];
#pragma unroll
        for (int j = 1; j < K; ++j) {  // SendBuf = sum_t GradBuf_t, in buffer order
            s.x += g[j].x;
            s.y += g[j].y;
            s.z += g[j].z;
            s.w += g[j].w;
        }
        float4 o;
        ps_apply1<OPT>(s.x, w.x, &st.x, eta, hp, wd, o.x);
        ps_apply1<OPT>(s.y, w.y, &st.y, eta, hp, wd, o.y);
        ps_apply1<OPT>(s.z, w.z, &st.z, eta, hp, wd, o.z);
        ps_apply1<OPT>(s.w, w.w, &st.w, eta, hp, wd, o.w);
        if constexpr (OPT != PS_SGD) st_stream(state + 4 * i, st);
        st_stream(w_out + 4 * i, o);
    }
    // scalar tail (n % 4 elements), handled by the first CTA
    if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
        const size_t i = 4 * n4 + threadIdx.x;
        float s = bufs.p[0][i];
        for (int j = 1; j < K; ++j) s += bufs.p[j][i];
        float st = (OPT != PS_SGD) ? state[i] : 0.f;
        float o;
        ps_apply1<OPT>(s, w_in[i], &st, eta, hp, wd, o);
        if constexpr (OPT != PS_SGD) state[i] = st;
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

// The same update over a row-major [rows][cols] weight matrix that also writes
// W' transposed (wT_out[c][r] = w_out[r][c]: the copy the input-gradient GEMMs
// read), instead of a separate transpose pass that would read W' back. A block
// takes a 32-row x 128-column tile: 8 warps, each thread one float4 column
// group of 4 of its rows (every warp access a 512-byte row segment); W' goes
// through shared memory and leaves as 32-float runs of W'^T rows. VEC: cols %
// 4 == 0 and 16-byte aligned pointers (float4 accesses), else scalar ones.
// The tile size also sets how the update shares the GPU with the tensor-core
// GEMMs it overlaps on another stream: with 16.5 KB of shared memory exactly one
// block fits beside a 256-wide pair GEMM CTA (~210 KB). Measured on the SMLPs
// step: no block beside a GEMM CTA (padded tile) 729k images/s, one 767k, two
// or more (32 x 32 tiles) 732k — more co-resident update blocks slow the GEMMs
// more than they gain, none leaves the update to the gaps between GEMMs.
constexpr int kUtRows = 32, kUtCols = 128;

template <int OPT, int K, bool VEC>
__global__ void __launch_bounds__(256) update_t_kernel(const float* w_in, float* w_out, float* wT_out, float* state,
                                                       BufPtrs bufs, int rows, int cols, size_t n_total, float eta,
                                                       float hp, float wd) {
    __shared__ float tile[kUtRows][kUtCols + 1];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int r0 = blockIdx.y * kUtRows, c0 = blockIdx.x * kUtCols;
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        // the elements after the matrix (a layer's bias): the flat update, no transpose
        for (size_t i = static_cast<size_t>(rows) * cols + threadIdx.x; i < n_total; i += blockDim.x) {
            float sm = bufs.p[0][i];
            for (int b = 1; b < K; ++b) sm += bufs.p[b][i];
            float st = (OPT != PS_SGD) ? state[i] : 0.f;
            float o;
            ps_apply1<OPT>(sm, w_in[i], &st, eta, hp, wd, o);
            if constexpr (OPT != PS_SGD) state[i] = st;
            w_out[i] = o;
        }
    }
#pragma unroll
    for (int j = 0; j < kUtRows / 8; ++j) {
        const int rr = ty + 8 * j, r = r0 + rr;
        const int c = c0 + 4 * tx;
        if (r >= rows) continue;
        const size_t off = static_cast<size_t>(r) * cols + c;
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        if (VEC && c + 4 <= cols) {
            float4 g[K];
#pragma unroll
            for (int b = 0; b < K; ++b) g[b] = ld_stream(bufs.p[b] + off);
            const float4 w = ld_stream(w_in + off);
            float4 st = make_float4(0.f, 0.f, 0.f, 0.f);
            if constexpr (OPT != PS_SGD) st = ld_stream(state + off);
            float4 sm = g[0];
#pragma unroll
            for (int b = 1; b < K; ++b) {  // SendBuf = sum_t GradBuf_t, in buffer order
                sm.x += g[b].x;
                sm.y += g[b].y;
                sm.z += g[b].z;
                sm.w += g[b].w;
            }
            ps_apply1<OPT>(sm.x, w.x, &st.x, eta, hp, wd, o[0]);
            ps_apply1<OPT>(sm.y, w.y, &st.y, eta, hp, wd, o[1]);
            ps_apply1<OPT>(sm.z, w.z, &st.z, eta, hp, wd, o[2]);
            ps_apply1<OPT>(sm.w, w.w, &st.w, eta, hp, wd, o[3]);
            if constexpr (OPT != PS_SGD) st_stream(state + off, st);
            st_stream(w_out + off, make_float4(o[0], o[1], o[2], o[3]));
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (c + e >= cols) break;
                float sm = bufs.p[0][off + e];
                for (int b = 1; b < K; ++b) sm += bufs.p[b][off + e];
                float st = (OPT != PS_SGD) ? state[off + e] : 0.f;
                ps_apply1<OPT>(sm, w_in[off + e], &st, eta, hp, wd, o[e]);
                if constexpr (OPT != PS_SGD) state[off + e] = st;
                w_out[off + e] = o[e];
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) tile[rr][4 * tx + e] = o[e];
    }
    __syncthreads();
    // W'^T rows c0.. (columns of W), 32 consecutive entries (rows of W) per warp store
#pragma unroll
    for (int j = 0; j < kUtCols / 8; ++j) {
        const int cc = ty + 8 * j, c = c0 + cc, r = r0 + tx;
        if (c < cols && r < rows) __stcs(wT_out + static_cast<size_t>(c) * rows + r, tile[tx][cc]);
    }
}

int stream_grid(size_t n) {
    const size_t n4 = n / 4 + 1;
    size_t want = (n4 + kThreads - 1) / kThreads;
    size_t cap = static_cast<size_t>(num_sms()) * 8;  // 8 x 256 threads per SM
    return static_cast<int>(want < cap ? want : cap);
}

template <int OPT>
int launch_update(const char* fn, const float* w_in, float* w_out, float* state, const float* const* bufs, int k,
                  size_t n, float eta, float hp, float wd, sprint_stream_t stream) {
    SPRINT_REQUIRE(k >= 1, SPRINT_ERR_SHAPE, "%s: k must be >= 1 (got %d)", fn, k);
    SPRINT_REQUIRE(k <= kMaxBufs, SPRINT_ERR_UNSUPPORTED, "%s: k = %d > %d buffers", fn, k, kMaxBufs);
    if (n == 0) return SPRINT_OK;
    SPRINT_REQUIRE(w_in && w_out && bufs, SPRINT_ERR_INVALID_ARG, "%s: NULL w_in, w_out or bufs", fn);
    SPRINT_REQUIRE(OPT == PS_SGD || state, SPRINT_ERR_INVALID_ARG, "%s: NULL optimizer state", fn);
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
    case KK: update_kernel<OPT, KK><<<grid, kThreads, 0, s>>>(w_in, w_out, state, bp, n, eta, hp, wd); break;
        SPRINT_K(1) SPRINT_K(2) SPRINT_K(3) SPRINT_K(4) SPRINT_K(5) SPRINT_K(6) SPRINT_K(7) SPRINT_K(8)
        SPRINT_K(9) SPRINT_K(10) SPRINT_K(11) SPRINT_K(12) SPRINT_K(13) SPRINT_K(14) SPRINT_K(15) SPRINT_K(16)
#undef SPRINT_K
    }
    return check_launch(fn);
}

template <int OPT>
int launch_update_t(const char* fn, const float* w_in, float* w_out, float* wT_out, float* state,
                    const float* const* bufs, int k, int rows, int cols, size_t n_total, float eta, float hp, float wd,
                    sprint_stream_t stream) {
    SPRINT_REQUIRE(k >= 1, SPRINT_ERR_SHAPE, "%s: k must be >= 1 (got %d)", fn, k);
    SPRINT_REQUIRE(k <= kMaxBufs, SPRINT_ERR_UNSUPPORTED, "%s: k = %d > %d buffers", fn, k, kMaxBufs);
    SPRINT_REQUIRE(rows >= 1 && cols >= 1, SPRINT_ERR_SHAPE, "%s: rows and cols must be >= 1 (got %d, %d)", fn, rows,
                   cols);
    SPRINT_REQUIRE(n_total >= static_cast<size_t>(rows) * cols, SPRINT_ERR_SHAPE,
                   "%s: n_total %zu is below rows * cols", fn, n_total);
    SPRINT_REQUIRE(rows <= 65535 * kUtRows, SPRINT_ERR_SHAPE, "%s: %d rows exceed the grid", fn, rows);
    SPRINT_REQUIRE(w_in && w_out && wT_out && bufs, SPRINT_ERR_INVALID_ARG, "%s: NULL w_in, w_out, wT_out or bufs",
                   fn);
    SPRINT_REQUIRE(OPT == PS_SGD || state, SPRINT_ERR_INVALID_ARG, "%s: NULL optimizer state", fn);
    BufPtrs bp{};
    bool vec = cols % 4 == 0 && aligned16(w_in) && aligned16(w_out) && (!state || aligned16(state));
    for (int j = 0; j < k; ++j) {
        SPRINT_REQUIRE(bufs[j], SPRINT_ERR_INVALID_ARG, "%s: bufs[%d] is NULL", fn, j);
        vec = vec && aligned16(bufs[j]);
        bp.p[j] = bufs[j];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 grid((cols + kUtCols - 1) / kUtCols, (rows + kUtRows - 1) / kUtRows);
    switch (k) {
#define SPRINT_K(KK)                                                                                            \
    case KK:                                                                                                    \
        if (vec)                                                                                                \
            update_t_kernel<OPT, KK, true><<<grid, 256, 0, s>>>(w_in, w_out, wT_out, state, bp, rows, cols, n_total, eta, hp, wd); \
        else                                                                                                    \
            update_t_kernel<OPT, KK, false><<<grid, 256, 0, s>>>(w_in, w_out, wT_out, state, bp, rows, cols, n_total, eta, hp, wd); \
        break;
        SPRINT_K(1) SPRINT_K(2) SPRINT_K(3) SPRINT_K(4) SPRINT_K(5) SPRINT_K(6) SPRINT_K(7) SPRINT_K(8)
        SPRINT_K(9) SPRINT_K(10) SPRINT_K(11) SPRINT_K(12) SPRINT_K(13) SPRINT_K(14) SPRINT_K(15) SPRINT_K(16)
#undef SPRINT_K
    }
    return check_launch(fn);
}

}  // namespace

// the standalone update by rule (PsOpt), for callers in other files
int launch_ps_update(int opt, const char* fn, const float* w_in, float* w_out, float* state, const float* const* bufs,
                     int k, size_t n, float eta, float hp, float wd, sprint_stream_t stream) {
    switch (opt) {
        case PS_SGD: return launch_update<PS_SGD>(fn, w_in, w_out, nullptr, bufs, k, n, eta, hp, wd, stream);
        case PS_MOMENTUM: return launch_update<PS_MOMENTUM>(fn, w_in, w_out, state, bufs, k, n, eta, hp, wd, stream);
        case PS_NESTEROV: return launch_update<PS_NESTEROV>(fn, w_in, w_out, state, bufs, k, n, eta, hp, wd, stream);
        case PS_ADAGRAD: return launch_update<PS_ADAGRAD>(fn, w_in, w_out, state, bufs, k, n, eta, hp, wd, stream);
        default: return fail(SPRINT_ERR_INVALID_ARG, "%s: unknown update rule %d", fn, opt);
    }
}

int launch_ps_update_t(int opt, const char* fn, const float* w_in, float* w_out, float* wT_out, float* state,
                       const float* const* bufs, int k, int rows, int cols, size_t n_total, float eta, float hp,
                       float wd, sprint_stream_t stream) {
    switch (opt) {
        case PS_SGD:
            return launch_update_t<PS_SGD>(fn, w_in, w_out, wT_out, nullptr, bufs, k, rows, cols, n_total, eta, hp,
                                           wd, stream);
        case PS_MOMENTUM:
            return launch_update_t<PS_MOMENTUM>(fn, w_in, w_out, wT_out, state, bufs, k, rows, cols, n_total, eta, hp,
                                                wd, stream);
        case PS_NESTEROV:
            return launch_update_t<PS_NESTEROV>(fn, w_in, w_out, wT_out, state, bufs, k, rows, cols, n_total, eta, hp,
                                                wd, stream);
        case PS_ADAGRAD:
            return launch_update_t<PS_ADAGRAD>(fn, w_in, w_out, wT_out, state, bufs, k, rows, cols, n_total, eta, hp,
                                               wd, stream);
        default: return fail(SPRINT_ERR_INVALID_ARG, "%s: unknown update rule %d", fn, opt);
    }
}

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
    return launch_update<PS_SGD>(__func__, w_in, w_out, nullptr, bufs, k, n, eta, 0.f, 0.f, stream);
}

extern "C" int sprint_apply_update_momentum(const float* w_in, float* w_out, float* v, const float* const* bufs, int k,
                                            size_t n, float eta, float nu, sprint_stream_t stream) {
    return launch_update<PS_MOMENTUM>(__func__, w_in, w_out, v, bufs, k, n, eta, nu, 0.f, stream);
}

extern "C" int sprint_apply_update_adagrad(const float* w_in, float* w_out, float* G, const float* const* bufs, int k,
                                           size_t n, float eta, float eps, sprint_stream_t stream) {
    return launch_update<PS_ADAGRAD>(__func__, w_in, w_out, G, bufs, k, n, eta, eps, 0.f, stream);
}

extern "C" int sprint_apply_update(int opt, const float* w_in, float* w_out, float* state, const float* const* bufs,
                                   int k, size_t n, float eta, float nu_or_eps, float weight_decay,
                                   sprint_stream_t stream) {
    return launch_ps_update(opt, __func__, w_in, w_out, state, bufs, k, n, eta, nu_or_eps, weight_decay, stream);
}

extern "C" int sprint_apply_update_t(int opt, const float* w_in, float* w_out, float* wT_out, float* state,
                                     const float* const* bufs, int k, int rows, int cols, size_t n_total, float eta,
                                     float nu_or_eps, float weight_decay, sprint_stream_t stream) {
    return launch_ps_update_t(opt, __func__, w_in, w_out, wT_out, state, bufs, k, rows, cols, n_total, eta, nu_or_eps,
                              weight_decay, stream);
}
