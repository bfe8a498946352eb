// Memory-bound layers of the worker step: 2x2 max-pool forward/backward
// ([S] Sec. 3.2, pooling p_l = 2), softmax cross-entropy (the softmax output
// layer), the explicit im2col of [S] Eq. (5), and the column reduction that
// forms dE/db (the "dedb" role, m = 1) with the GradBuf accumulate fused.
#include "common.cuh"

namespace sprint {

// Column sums with the GradBuf epilogue: out[c] = (accumulate ? out[c] : 0) + alpha * sum_r in[r*cols + c].
// Launched as (ceil(cols/32), chunks) blocks of 32x8 threads. With chunks == 1
// the epilogue is applied directly; otherwise each chunk writes its partial
// sum to partial[chunk*cols + c] and colsum_finish adds them in chunk order.
__global__ void __launch_bounds__(256) colsum_kernel(const float* __restrict__ in, long long rows, int cols,
                                                     long long rows_per_chunk, float* __restrict__ partial,
                                                     float* __restrict__ out, float alpha, int accumulate) {
    __shared__ float red[8][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + tx;
    const long long r0 = static_cast<long long>(blockIdx.y) * rows_per_chunk;
    long long r1 = r0 + rows_per_chunk;
    if (r1 > rows) r1 = rows;
    float s = 0.f;
    if (c < cols)
        for (long long r = r0 + ty; r < r1; r += 8) s += in[r * cols + c];
    red[ty][tx] = s;
    __syncthreads();
    if (ty == 0 && c < cols) {
        float t = red[0][tx];
#pragma unroll
        for (int k = 1; k < 8; ++k) t += red[k][tx];
        if (gridDim.y == 1)
            out[c] = (accumulate ? out[c] : 0.f) + alpha * t;
        else
            partial[static_cast<long long>(blockIdx.y) * cols + c] = t;
    }
}

__global__ void colsum_finish(const float* __restrict__ partial, int chunks, int cols, float* __restrict__ out,
                              float alpha, int accumulate) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= cols) return;
    const float t = ordered_strided_sum(partial + c, chunks, cols);
    out[c] = (accumulate ? out[c] : 0.f) + alpha * t;
}

// Column sums for cols % 4 == 0: a block of 32 x 32 threads covers 128 columns
// (tx: a float4 of 4 columns) and one chunk of rows (ty: every 32nd row, four
// independent loads in flight per thread); the 32 row stripes are then added
// in stripe order. Same epilogue / partial convention as colsum_kernel.
__global__ void __launch_bounds__(1024) colsum4_kernel(const float* __restrict__ in, long long rows, int cols,
                                                       long long rows_per_chunk, float* __restrict__ partial,
                                                       float* __restrict__ out, float alpha, int accumulate) {
    __shared__ float4 red[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int col = (blockIdx.x * 32 + tx) * 4;
    const long long r0 = static_cast<long long>(blockIdx.y) * rows_per_chunk;
    long long r1 = r0 + rows_per_chunk;
    if (r1 > rows) r1 = rows;
    float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0, s2 = s0, s3 = s0;
    if (col < cols) {
        const float* base = in + col;
        long long r = r0 + ty;
        for (; r + 96 < r1; r += 128) {
            const float4 a = *reinterpret_cast<const float4*>(base + r * cols);
            const float4 b = *reinterpret_cast<const float4*>(base + (r + 32) * cols);
            const float4 c = *reinterpret_cast<const float4*>(base + (r + 64) * cols);
            const float4 d = *reinterpret_cast<const float4*>(base + (r + 96) * cols);
            s0.x += a.x; s0.y += a.y; s0.z += a.z; s0.w += a.w;
            s1.x += b.x; s1.y += b.y; s1.z += b.z; s1.w += b.w;
            s2.x += c.x; s2.y += c.y; s2.z += c.z; s2.w += c.w;
            s3.x += d.x; s3.y += d.y; s3.z += d.z; s3.w += d.w;
        }
        for (; r < r1; r += 32) {
            const float4 a = *reinterpret_cast<const float4*>(base + r * cols);
            s0.x += a.x; s0.y += a.y; s0.z += a.z; s0.w += a.w;
        }
    }
    red[ty][tx] = make_float4(s0.x + s1.x + s2.x + s3.x, s0.y + s1.y + s2.y + s3.y, s0.z + s1.z + s2.z + s3.z,
                              s0.w + s1.w + s2.w + s3.w);
    __syncthreads();
    if (ty == 0 && col < cols) {
        float4 t = red[0][tx];
        for (int k = 1; k < 32; ++k) {
            const float4 u = red[k][tx];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        if (gridDim.y == 1) {
            float4 o = make_float4(alpha * t.x, alpha * t.y, alpha * t.z, alpha * t.w);
            if (accumulate) {
                const float4 prev = *reinterpret_cast<const float4*>(out + col);
                o.x += prev.x; o.y += prev.y; o.z += prev.z; o.w += prev.w;
            }
            *reinterpret_cast<float4*>(out + col) = o;
        } else {
            *reinterpret_cast<float4*>(partial + static_cast<long long>(blockIdx.y) * cols + col) = t;
        }
    }
}

// Number of chunks colsum uses for `rows` rows (1 means no workspace).
int colsum_chunks(long long rows, int cols) {
    if (rows <= 8192) return 1;
    const long long col_blocks = (cols + 127) / 128;
    long long want = (2ll * num_sms() + col_blocks - 1) / col_blocks;   // ~2 blocks per SM
    const long long by_rows = rows / 1024;
    if (want > by_rows) want = by_rows;
    if (want < 1) want = 1;
    return static_cast<int>(want);
}

// With partial == nullptr the sum runs as one chunk (no workspace).
int launch_colsum(const float* in, long long rows, int cols, float* partial, float* out, float alpha, int accumulate,
                  cudaStream_t s) {
    const int chunks = partial ? colsum_chunks(rows, cols) : 1;
    const long long per = (rows + chunks - 1) / chunks;
    const bool vec = (cols % 4 == 0) && aligned16(in) && aligned16(out) && (!partial || aligned16(partial));
    if (vec) {
        dim3 grid((cols + 127) / 128, chunks);
        colsum4_kernel<<<grid, 1024, 0, s>>>(in, rows, cols, per, partial, out, alpha, accumulate);
    } else {
        dim3 grid((cols + 31) / 32, chunks);
        colsum_kernel<<<grid, 256, 0, s>>>(in, rows, cols, per, partial, out, alpha, accumulate);
    }
    if (chunks > 1) colsum_finish<<<(cols + 127) / 128, 128, 0, s>>>(partial, chunks, cols, out, alpha, accumulate);
    return check_launch("colsum", chunks > 1 ? 2 : 1);
}

// Strided batched transpose through 32x32 shared-memory tiles, coalesced on
// both sides: dst[b*db + c*dc + (r/32)*drt + r%32] = src[b*sb + r*sr + c] for
// r < R, c < C, b = blockIdx.z (drt = 32: dst[b*db + c*dc + r]). Used for
// w -> w^T (one batch), NHWC -> [C][H][W][N] (batch = pixel) and NHWC ->
// [H][W*N/32][C][32] (batch = pixel, dc = 32, drt = 32*C). A block takes CT
// tiles side by side along c (2 for C >= 64, 4 for C >= 128), so that each
// thread has 4 * CT loads in flight: the copy is bound by the bytes in flight.
template <int CT>
__global__ void __launch_bounds__(256) transpose_kernel(const float* __restrict__ src, float* __restrict__ dst, int R,
                                                        int C, long long sb, long long sr, long long db, long long dc,
                                                        long long drt) {
    __shared__ float tile[CT][32][33];
    const long long b = blockIdx.z;
    const int r0 = blockIdx.y * 32, cb = blockIdx.x * 32 * CT;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
    for (int ct = 0; ct < CT; ++ct)
#pragma unroll
        for (int j = ty; j < 32; j += 8) {
            const int r = r0 + j, c = cb + 32 * ct + tx;
            if (r < R && c < C) tile[ct][j][tx] = src[b * sb + static_cast<long long>(r) * sr + c];
        }
    __syncthreads();
    const long long dst0 = b * db + blockIdx.y * drt;
#pragma unroll
    for (int ct = 0; ct < CT; ++ct)
#pragma unroll
        for (int j = ty; j < 32; j += 8) {
            const int c = cb + 32 * ct + j, r = r0 + tx;
            if (r < R && c < C) dst[dst0 + static_cast<long long>(c) * dc + tx] = tile[ct][tx][j];
        }
}

int launch_transpose(const float* src, float* dst, int batch, int R, int C, long long sb, long long sr, long long db,
                     long long dc, cudaStream_t s, long long drt = 32) {
    if (batch <= 0 || R <= 0 || C <= 0) return SPRINT_OK;
    if (batch > 65535 || (R + 31) / 32 > 65535)
        return fail(SPRINT_ERR_SHAPE, "transpose: batch %d / rows %d exceed the grid limits", batch, R);
    if (C >= 128) {
        dim3 grid((C + 127) / 128, (R + 31) / 32, batch);
        transpose_kernel<4><<<grid, 256, 0, s>>>(src, dst, R, C, sb, sr, db, dc, drt);
    } else if (C >= 64) {
        dim3 grid((C + 63) / 64, (R + 31) / 32, batch);
        transpose_kernel<2><<<grid, 256, 0, s>>>(src, dst, R, C, sb, sr, db, dc, drt);
    } else {
        dim3 grid((C + 31) / 32, (R + 31) / 32, batch);
        transpose_kernel<1><<<grid, 256, 0, s>>>(src, dst, R, C, sb, sr, db, dc, drt);
    }
    return check_launch("transpose_kernel");
}

// transpose_kernel plus the column sums the dedb role needs from the same
// tile: after the transpose, the block's 32 rows (images) of each of its 32
// columns (channels) are added in row order into partial[c * nparts + part],
// part = batch index * row tiles + row tile; colsum_parts_finish then adds a
// channel's parts in part order. One read of dy serves both dy^T and dedb.
template <int CT>
__global__ void __launch_bounds__(256) transpose_colsum_kernel(const float* __restrict__ src, float* __restrict__ dst,
                                                               int R, int C, long long sb, long long sr, long long db,
                                                               long long dc, long long drt, float* __restrict__ partial,
                                                               long long nparts) {
    __shared__ float tile[CT][32][33];
    const long long b = blockIdx.z;
    const int r0 = blockIdx.y * 32, cb = blockIdx.x * 32 * CT;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
    for (int ct = 0; ct < CT; ++ct)
#pragma unroll
        for (int j = ty; j < 32; j += 8) {
            const int r = r0 + j, c = cb + 32 * ct + tx;
            tile[ct][j][tx] = (r < R && c < C) ? src[b * sb + static_cast<long long>(r) * sr + c] : 0.f;
        }
    __syncthreads();
    const long long dst0 = b * db + blockIdx.y * drt;
#pragma unroll
    for (int ct = 0; ct < CT; ++ct)
#pragma unroll
        for (int j = ty; j < 32; j += 8) {
            const int c = cb + 32 * ct + j, r = r0 + tx;
            if (r < R && c < C) dst[dst0 + static_cast<long long>(c) * dc + tx] = tile[ct][tx][j];
        }
    if (ty < CT && cb + 32 * ty + tx < C) {   // warp ct adds sub-tile ct's columns
        float t = 0.f;
        for (int j = 0; j < 32; ++j) t += tile[ty][j][tx];
        partial[static_cast<long long>(cb + 32 * ty + tx) * nparts + b * gridDim.y + blockIdx.y] = t;
    }
}

// out[c] = (accumulate ? out[c] : 0) + alpha * sum over the nparts parts of
// channel c, added as 256 thread stripes (part = t, t + 256, ...) and then a
// fixed pairwise tree: the same order on every run.
__global__ void __launch_bounds__(256) colsum_parts_finish(const float* __restrict__ partial, long long nparts,
                                                           float* __restrict__ out, float alpha, int accumulate) {
    __shared__ float red[256];
    const int c = blockIdx.x;
    const float* p = partial + static_cast<long long>(c) * nparts;
    const float t = threadIdx.x < nparts
                        ? ordered_strided_sum(p + threadIdx.x, static_cast<int>((nparts - threadIdx.x + 255) / 256), 256)
                        : 0.f;
    red[threadIdx.x] = t;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) out[c] = (accumulate ? out[c] : 0.f) + alpha * red[0];
}

// dst = src transposed as launch_transpose does, and out = dedb of src's columns
// (partial: C * batch * ceil(R / 32) floats of workspace)
int launch_transpose_colsum(const float* src, float* dst, int batch, int R, int C, long long sb, long long sr,
                            long long db, long long dc, float* partial, float* out, float alpha, int accumulate,
                            cudaStream_t s, long long drt = 32) {
    if (batch <= 0 || R <= 0 || C <= 0) return SPRINT_OK;
    if (batch > 65535 || (R + 31) / 32 > 65535)
        return fail(SPRINT_ERR_SHAPE, "transpose: batch %d / rows %d exceed the grid limits", batch, R);
    const long long nparts = static_cast<long long>(batch) * ((R + 31) / 32);
    if (C >= 128) {
        dim3 grid((C + 127) / 128, (R + 31) / 32, batch);
        transpose_colsum_kernel<4><<<grid, 256, 0, s>>>(src, dst, R, C, sb, sr, db, dc, drt, partial, nparts);
    } else if (C >= 64) {
        dim3 grid((C + 63) / 64, (R + 31) / 32, batch);
        transpose_colsum_kernel<2><<<grid, 256, 0, s>>>(src, dst, R, C, sb, sr, db, dc, drt, partial, nparts);
    } else {
        dim3 grid((C + 31) / 32, (R + 31) / 32, batch);
        transpose_colsum_kernel<1><<<grid, 256, 0, s>>>(src, dst, R, C, sb, sr, db, dc, drt, partial, nparts);
    }
    colsum_parts_finish<<<C, 256, 0, s>>>(partial, nparts, out, alpha, accumulate);
    return check_launch("transpose_colsum", 2);
}

// One launch over up to kMaxGroup problems (blockIdx.z = problem g):
// out[g] = in[g]^T, in[g] being R x C row-major.
struct GroupPtrs {
    const float* in[kMaxGroup];
    float* out[kMaxGroup];
};

__global__ void __launch_bounds__(256) transpose_group_kernel(GroupPtrs t, int R, int C) {
    __shared__ float tile[32][33];
    const float* __restrict__ src = t.in[blockIdx.z];
    float* __restrict__ dst = t.out[blockIdx.z];
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
    for (int j = ty; j < 32; j += 8) {
        const int r = r0 + j, c = c0 + tx;
        if (r < R && c < C) tile[j][tx] = src[static_cast<long long>(r) * C + c];
    }
    __syncthreads();
#pragma unroll
    for (int j = ty; j < 32; j += 8) {
        const int c = c0 + j, r = r0 + tx;
        if (r < R && c < C) dst[static_cast<long long>(c) * R + r] = tile[tx][j];
    }
}

int launch_transpose_group(const float* const* src, float* const* dst, int G, int R, int C, cudaStream_t s) {
    if (G <= 0 || R <= 0 || C <= 0) return SPRINT_OK;
    if ((R + 31) / 32 > 65535) return fail(SPRINT_ERR_SHAPE, "transpose: %d rows exceed the grid limits", R);
    for (int g0 = 0; g0 < G; g0 += kMaxGroup) {
        const int n = G - g0 < kMaxGroup ? G - g0 : kMaxGroup;
        GroupPtrs t{};
        for (int i = 0; i < n; ++i) {
            t.in[i] = src[g0 + i];
            t.out[i] = dst[g0 + i];
        }
        transpose_group_kernel<<<dim3((C + 31) / 32, (R + 31) / 32, n), 256, 0, s>>>(t, R, C);
        int rc = check_launch("transpose_group_kernel");
        if (rc) return rc;
    }
    return SPRINT_OK;
}

// Column sums of up to kMaxGroup row-major [rows][cols] matrices (cols % 4 == 0,
// one chunk of rows: the FC bias gradient), blockIdx.y = problem; same
// arithmetic order and epilogue as colsum4_kernel with one chunk.
__global__ void __launch_bounds__(1024) colsum4_group_kernel(GroupPtrs t, long long rows, int cols, float alpha,
                                                             int accumulate) {
    __shared__ float4 red[32][33];
    const float* __restrict__ in = t.in[blockIdx.y];
    float* __restrict__ out = t.out[blockIdx.y];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int col = (blockIdx.x * 32 + tx) * 4;
    float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0, s2 = s0, s3 = s0;
    if (col < cols) {
        const float* base = in + col;
        long long r = ty;
        for (; r + 96 < rows; r += 128) {
            const float4 a = *reinterpret_cast<const float4*>(base + r * cols);
            const float4 b = *reinterpret_cast<const float4*>(base + (r + 32) * cols);
            const float4 c = *reinterpret_cast<const float4*>(base + (r + 64) * cols);
            const float4 d = *reinterpret_cast<const float4*>(base + (r + 96) * cols);
            s0.x += a.x; s0.y += a.y; s0.z += a.z; s0.w += a.w;
            s1.x += b.x; s1.y += b.y; s1.z += b.z; s1.w += b.w;
            s2.x += c.x; s2.y += c.y; s2.z += c.z; s2.w += c.w;
            s3.x += d.x; s3.y += d.y; s3.z += d.z; s3.w += d.w;
        }
        for (; r < rows; r += 32) {
            const float4 a = *reinterpret_cast<const float4*>(base + r * cols);
            s0.x += a.x; s0.y += a.y; s0.z += a.z; s0.w += a.w;
        }
    }
    red[ty][tx] = make_float4(s0.x + s1.x + s2.x + s3.x, s0.y + s1.y + s2.y + s3.y, s0.z + s1.z + s2.z + s3.z,
                              s0.w + s1.w + s2.w + s3.w);
    __syncthreads();
    if (ty == 0 && col < cols) {
        float4 u = red[0][tx];
        for (int k = 1; k < 32; ++k) {
            const float4 v = red[k][tx];
            u.x += v.x; u.y += v.y; u.z += v.z; u.w += v.w;
        }
        float4 o = make_float4(alpha * u.x, alpha * u.y, alpha * u.z, alpha * u.w);
        if (accumulate) {
            const float4 prev = *reinterpret_cast<const float4*>(out + col);
            o.x += prev.x; o.y += prev.y; o.z += prev.z; o.w += prev.w;
        }
        *reinterpret_cast<float4*>(out + col) = o;
    }
}

// Narrow column sums (cols <= 16, e.g. a classifier's bias gradient), one
// block per problem (blockIdx.x): thread t adds rows t, t+256, ... for every
// column, then the 256 partial sums of a column are added in thread order.
__global__ void __launch_bounds__(256) colsum_narrow_group_kernel(GroupPtrs t, long long rows, int cols, float alpha,
                                                                  int accumulate) {
    __shared__ float red[16][257];
    const float* __restrict__ in = t.in[blockIdx.x];
    float* __restrict__ out = t.out[blockIdx.x];
    float acc[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = 0.f;
    for (long long r = threadIdx.x; r < rows; r += 256) {
        const float* row = in + r * cols;
#pragma unroll
        for (int c = 0; c < 16; ++c)
            if (c < cols) acc[c] += row[c];
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) red[c][threadIdx.x] = acc[c];
    __syncthreads();
    if (threadIdx.x < cols) {
        const int c = threadIdx.x;
        float s = 0.f;
        for (int i = 0; i < 256; ++i) s += red[c][i];
        out[c] = (accumulate ? out[c] : 0.f) + alpha * s;
    }
}

// out[g][c] = (accumulate ? out[g][c] : 0) + alpha * sum_r in[g][r][c], one chunk per problem
int launch_colsum_group(const float* const* in, float* const* out, int G, long long rows, int cols, float alpha,
                        int accumulate, cudaStream_t s) {
    bool vec = cols % 4 == 0;
    for (int g = 0; g < G && vec; ++g) vec = aligned16(in[g]) && aligned16(out[g]);
    if (!vec && cols <= 16) {
        for (int g0 = 0; g0 < G; g0 += kMaxGroup) {
            const int n = G - g0 < kMaxGroup ? G - g0 : kMaxGroup;
            GroupPtrs t{};
            for (int i = 0; i < n; ++i) {
                t.in[i] = in[g0 + i];
                t.out[i] = out[g0 + i];
            }
            colsum_narrow_group_kernel<<<n, 256, 0, s>>>(t, rows, cols, alpha, accumulate);
            const int rc = check_launch("colsum_narrow_group_kernel");
            if (rc) return rc;
        }
        return SPRINT_OK;
    }
    if (!vec) {
        for (int g = 0; g < G; ++g) {
            const int rc = launch_colsum(in[g], rows, cols, nullptr, out[g], alpha, accumulate, s);
            if (rc) return rc;
        }
        return SPRINT_OK;
    }
    for (int g0 = 0; g0 < G; g0 += kMaxGroup) {
        const int n = G - g0 < kMaxGroup ? G - g0 : kMaxGroup;
        GroupPtrs t{};
        for (int i = 0; i < n; ++i) {
            t.in[i] = in[g0 + i];
            t.out[i] = out[g0 + i];
        }
        colsum4_group_kernel<<<dim3((cols + 127) / 128, n), 1024, 0, s>>>(t, rows, cols, alpha, accumulate);
        const int rc = check_launch("colsum4_group_kernel");
        if (rc) return rc;
    }
    return SPRINT_OK;
}

namespace {

// ------------------------------------------------------------------ pooling
template <int V>
__global__ void __launch_bounds__(256) pool_fwd_kernel(const float* __restrict__ x, float* __restrict__ y,
                                                       uint8_t* __restrict__ arg, int N, int H, int W, int C) {
    const int Ho = H / 2, Wo = W / 2, Cv = C / V;
    const long long total = static_cast<long long>(N) * Ho * Wo * Cv;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int cv = static_cast<int>(idx % Cv);
        long long p = idx / Cv;
        const int ow = static_cast<int>(p % Wo);
        p /= Wo;
        const int oh = static_cast<int>(p % Ho);
        const long long n = p / Ho;
        const long long base = ((n * H + 2 * oh) * W + 2 * ow) * C + static_cast<long long>(cv) * V;
        const long long ob = ((n * Ho + oh) * Wo + ow) * C + static_cast<long long>(cv) * V;
        const long long off[4] = {0, C, static_cast<long long>(W) * C, static_cast<long long>(W) * C + C};
        if constexpr (V == 4) {
            float4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] = *reinterpret_cast<const float4*>(x + base + off[q]);
            float b[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
            uint8_t a[4] = {0, 0, 0, 0};
#pragma unroll
            for (int q = 1; q < 4; ++q) {
                const float e[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                for (int l = 0; l < 4; ++l)
                    if (e[l] > b[l]) {  // strict: the first maximum in row-major order wins
                        b[l] = e[l];
                        a[l] = static_cast<uint8_t>(q);
                    }
            }
            *reinterpret_cast<float4*>(y + ob) = make_float4(b[0], b[1], b[2], b[3]);
            *reinterpret_cast<uchar4*>(arg + ob) = make_uchar4(a[0], a[1], a[2], a[3]);
        } else {
            float b = x[base];
            uint8_t a = 0;
#pragma unroll
            for (int q = 1; q < 4; ++q) {
                const float e = x[base + off[q]];
                if (e > b) {
                    b = e;
                    a = static_cast<uint8_t>(q);
                }
            }
            y[ob] = b;
            arg[ob] = a;
        }
    }
}

template <int V>
__global__ void __launch_bounds__(256) pool_bwd_kernel(const float* __restrict__ dy, const uint8_t* __restrict__ arg,
                                                       const float* __restrict__ pooled, float* __restrict__ dx, int N,
                                                       int H, int W, int C) {
    const int Ho = H / 2, Wo = W / 2, Cv = C / V;
    const long long total = static_cast<long long>(N) * Ho * Wo * Cv;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int cv = static_cast<int>(idx % Cv);
        long long p = idx / Cv;
        const int ow = static_cast<int>(p % Wo);
        p /= Wo;
        const int oh = static_cast<int>(p % Ho);
        const long long n = p / Ho;
        const long long base = ((n * H + 2 * oh) * W + 2 * ow) * C + static_cast<long long>(cv) * V;
        const long long ob = ((n * Ho + oh) * Wo + ow) * C + static_cast<long long>(cv) * V;
        const long long off[4] = {0, C, static_cast<long long>(W) * C, static_cast<long long>(W) * C + C};
        if constexpr (V == 4) {
            float4 g = *reinterpret_cast<const float4*>(dy + ob);
            const uchar4 a = *reinterpret_cast<const uchar4*>(arg + ob);
            if (pooled) {
                const float4 m = *reinterpret_cast<const float4*>(pooled + ob);
                g.x = m.x > 0.f ? g.x : 0.f;
                g.y = m.y > 0.f ? g.y : 0.f;
                g.z = m.z > 0.f ? g.z : 0.f;
                g.w = m.w > 0.f ? g.w : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float4 o;
                o.x = a.x == q ? g.x : 0.f;
                o.y = a.y == q ? g.y : 0.f;
                o.z = a.z == q ? g.z : 0.f;
                o.w = a.w == q ? g.w : 0.f;
                *reinterpret_cast<float4*>(dx + base + off[q]) = o;
            }
        } else {
            float g = dy[ob];
            if (pooled && !(pooled[ob] > 0.f)) g = 0.f;
            const uint8_t a = arg[ob];
#pragma unroll
            for (int q = 0; q < 4; ++q) dx[base + off[q]] = (a == q) ? g : 0.f;
        }
    }
}

// zeroes the trailing odd row (H odd) and column (W odd) that the pool ignores
__global__ void pool_bwd_edges(float* __restrict__ dx, int N, int H, int W, int C) {
    const long long row_elems = (H & 1) ? static_cast<long long>(W) * C : 0;
    const long long col_elems = (W & 1) ? static_cast<long long>(H) * C : 0;
    const long long per_img = row_elems + col_elems;
    const long long total = per_img * N;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long n = idx / per_img;
        long long r = idx % per_img;
        long long off;
        if (r < row_elems) {
            off = (n * H + (H - 1)) * static_cast<long long>(W) * C + r;
        } else {
            r -= row_elems;
            const long long h = r / C, c = r % C;
            off = ((n * H + h) * W + (W - 1)) * static_cast<long long>(C) + c;
        }
        dx[off] = 0.f;
    }
}

int grid_for(long long work, int threads = 256) {
    long long g = (work + threads - 1) / threads;
    const long long cap = static_cast<long long>(num_sms()) * 16;
    if (g > cap) g = cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

// ------------------------------------------------------------------ softmax
// One CTA; warp w handles rows w, w+32, ... Per-row losses are added in row
// order within a warp and the 32 warp sums in warp order, so the loss is
// deterministic.
// one problem per block: blockIdx.x selects the replica's tensors
struct XentTable {
    const float* logits[kMaxGroup];
    const int32_t* labels[kMaxGroup];
    float* loss[kMaxGroup];
    float* dlogits[kMaxGroup];
};

// A label outside [0, C) is not read through: that row's loss and gradient are
// zero and DEV_FLAG_BAD_LABEL is set in the device status word.
__global__ void __launch_bounds__(1024) softmax_xent_kernel(XentTable tab, int N, int C, float scale, int* status) {
    const float* logits = tab.logits[blockIdx.x];
    const int32_t* __restrict__ labels = tab.labels[blockIdx.x];
    float* __restrict__ loss = tab.loss[blockIdx.x];
    float* dlogits = tab.dlogits[blockIdx.x];
    __shared__ float warp_loss[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float acc = 0.f;
    for (int r = warp; r < N; r += 32) {
        const float* z = logits + static_cast<long long>(r) * C;
        float m = -INFINITY;
        for (int c = lane; c < C; c += 32) m = fmaxf(m, z[c]);
#pragma unroll
        for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float s = 0.f;
        for (int c = lane; c < C; c += 32) s += expf(z[c] - m);
#pragma unroll
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const int y = labels[r];
        const bool ok = y >= 0 && y < C;
        if (!ok && lane == 0 && status) atomicOr(status, DEV_FLAG_BAD_LABEL);
        const float zy = ok ? z[y] : 0.f;
        const float lse = m + logf(s);
        const float inv = 1.f / s;
        float* d = dlogits + static_cast<long long>(r) * C;
        __syncwarp();
        for (int c = lane; c < C; c += 32) {
            const float p = expf(z[c] - m) * inv;
            d[c] = ok ? (p - (c == y ? 1.f : 0.f)) * scale : 0.f;
        }
        __syncwarp();
        if (ok) acc += lse - zy;
    }
    if (lane == 0) warp_loss[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 32; ++w) t += warp_loss[w];
        *loss = t * scale;
    }
}

// Few classes (C <= 32): one row per thread; per-row losses are added by each
// warp in row order and the warp sums in warp order (deterministic).
__global__ void __launch_bounds__(1024) softmax_xent_rows_kernel(XentTable tab, int N, int C, float scale,
                                                                  int* status) {
    const float* logits = tab.logits[blockIdx.x];
    const int32_t* __restrict__ labels = tab.labels[blockIdx.x];
    float* __restrict__ loss = tab.loss[blockIdx.x];
    float* dlogits = tab.dlogits[blockIdx.x];
    __shared__ float warp_loss[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float acc = 0.f;
    for (int base = 0; base < N; base += 1024) {
        const int r = base + threadIdx.x;
        float row_loss = 0.f;
        if (r < N) {
            const float* z = logits + static_cast<long long>(r) * C;
            float* d = dlogits + static_cast<long long>(r) * C;
            float m = -INFINITY;
            for (int c = 0; c < C; ++c) m = fmaxf(m, z[c]);
            float s = 0.f;
            for (int c = 0; c < C; ++c) s += expf(z[c] - m);
            const int y = labels[r];
            if (y >= 0 && y < C) {
                const float zy = z[y];
                const float inv = 1.f / s;
                row_loss = m + logf(s) - zy;
                for (int c = 0; c < C; ++c) d[c] = (expf(z[c] - m) * inv - (c == y ? 1.f : 0.f)) * scale;
            } else {   // a label outside [0, C): not read through
                if (status) atomicOr(status, DEV_FLAG_BAD_LABEL);
                for (int c = 0; c < C; ++c) d[c] = 0.f;
            }
        }
        // add this pass's 32 rows of the warp in row order
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, row_loss, o);
            if (lane >= o) row_loss += t;
        }
        acc += __shfl_sync(0xffffffffu, row_loss, 31);
    }
    if (lane == 0) warp_loss[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 32; ++w) t += warp_loss[w];
        *loss = t * scale;
    }
}

// ------------------------------------------------------------------ im2col
template <int V>
__global__ void __launch_bounds__(256) im2col_kernel(const float* __restrict__ x, int N, int H, int W, int C, int pad,
                                                     float* __restrict__ col, int32_t* __restrict__ src) {
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    const int Kv = 9 * C / V, Cv = C / V;
    const long long total = static_cast<long long>(N) * Ho * Wo * Kv;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int kv = static_cast<int>(idx % Kv);
        long long p = idx / Kv;  // output pixel (n, oh, ow)
        const int ow = static_cast<int>(p % Wo);
        const long long q = p / Wo;
        const int oh = static_cast<int>(q % Ho);
        const long long n = q / Ho;
        const int tap = kv / Cv, ci = (kv % Cv) * V;
        const int ih = oh + tap / 3 - pad, iw = ow + tap % 3 - pad;
        const bool in = ih >= 0 && ih < H && iw >= 0 && iw < W;
        const long long s0 = ((n * H + ih) * W + iw) * C + ci;
        const long long d0 = p * 9 * C + static_cast<long long>(tap) * C + ci;
        if constexpr (V == 4) {
            const float4 v = in ? *reinterpret_cast<const float4*>(x + s0) : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(col + d0) = v;
            if (src) {
                const int b = in ? static_cast<int>(s0) : -1;
                *reinterpret_cast<int4*>(src + d0) = in ? make_int4(b, b + 1, b + 2, b + 3) : make_int4(-1, -1, -1, -1);
            }
        } else {
            col[d0] = in ? x[s0] : 0.f;
            if (src) src[d0] = in ? static_cast<int32_t>(s0) : -1;
        }
    }
}

}  // namespace
}  // namespace sprint

using namespace sprint;

extern "C" int sprint_pool_fwd(const float* x, float* y, uint8_t* argmax, int N, int H, int W, int C,
                               sprint_stream_t stream) {
    SPRINT_REQUIRE(N >= 1 && H >= 2 && W >= 2 && C >= 1, SPRINT_ERR_SHAPE, "%s: bad shape N=%d H=%d W=%d C=%d", __func__,
                   N, H, W, C);
    SPRINT_NONNULL(x, "x");
    SPRINT_NONNULL(y, "y");
    SPRINT_NONNULL(argmax, "argmax");
    SPRINT_ALIGNED(x, "x");
    SPRINT_ALIGNED(y, "y");
    SPRINT_ALIGNED(argmax, "argmax");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long outs = static_cast<long long>(N) * (H / 2) * (W / 2) * C;
    if (C % 4 == 0)
        pool_fwd_kernel<4><<<grid_for(outs / 4), 256, 0, s>>>(x, y, argmax, N, H, W, C);
    else
        pool_fwd_kernel<1><<<grid_for(outs), 256, 0, s>>>(x, y, argmax, N, H, W, C);
    return check_launch(__func__);
}

extern "C" int sprint_pool_bwd(const float* dy, const uint8_t* argmax, const float* pooled, float* dx, int N, int H,
                               int W, int C, sprint_stream_t stream) {
    SPRINT_REQUIRE(N >= 1 && H >= 2 && W >= 2 && C >= 1, SPRINT_ERR_SHAPE, "%s: bad shape N=%d H=%d W=%d C=%d", __func__,
                   N, H, W, C);
    SPRINT_NONNULL(dy, "dy");
    SPRINT_NONNULL(argmax, "argmax");
    SPRINT_NONNULL(dx, "dx");
    SPRINT_ALIGNED(dy, "dy");
    SPRINT_ALIGNED(argmax, "argmax");
    SPRINT_ALIGNED(pooled, "pooled");
    SPRINT_ALIGNED(dx, "dx");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long outs = static_cast<long long>(N) * (H / 2) * (W / 2) * C;
    if (C % 4 == 0)
        pool_bwd_kernel<4><<<grid_for(outs / 4), 256, 0, s>>>(dy, argmax, pooled, dx, N, H, W, C);
    else
        pool_bwd_kernel<1><<<grid_for(outs), 256, 0, s>>>(dy, argmax, pooled, dx, N, H, W, C);
    const bool odd = (H & 1) || (W & 1);
    if (odd) {
        const long long edge = static_cast<long long>(N) * (((H & 1) ? W : 0) + ((W & 1) ? H : 0)) * C;
        pool_bwd_edges<<<grid_for(edge), 256, 0, s>>>(dx, N, H, W, C);
    }
    return check_launch(__func__, odd ? 2 : 1);
}

namespace sprint {
namespace {
int launch_xent(const float* const* logits, const int32_t* const* labels, float* const* loss, float* const* dlogits,
                int G, int N, int C, int reduction_sum, cudaStream_t s) {
    const float scale = reduction_sum ? 1.f : 1.f / static_cast<float>(N);
    for (int g0 = 0; g0 < G; g0 += kMaxGroup) {
        const int n = G - g0 < kMaxGroup ? G - g0 : kMaxGroup;
        XentTable t{};
        for (int i = 0; i < n; ++i) {
            t.logits[i] = logits[g0 + i];
            t.labels[i] = labels[g0 + i];
            t.loss[i] = loss[g0 + i];
            t.dlogits[i] = dlogits[g0 + i];
        }
        if (C <= 32)
            softmax_xent_rows_kernel<<<n, 1024, 0, s>>>(t, N, C, scale, device_status_ptr());
        else
            softmax_xent_kernel<<<n, 1024, 0, s>>>(t, N, C, scale, device_status_ptr());
        const int rc = check_launch("softmax_xent");
        if (rc) return rc;
    }
    return SPRINT_OK;
}
}  // namespace
}  // namespace sprint

extern "C" int sprint_softmax_xent(const float* logits, const int32_t* labels, int N, int C, float* loss,
                                   float* dlogits, int reduction_sum, sprint_stream_t stream) {
    SPRINT_REQUIRE(N >= 1 && C >= 1, SPRINT_ERR_SHAPE, "%s: need N >= 1 and C >= 1 (got %d, %d)", __func__, N, C);
    SPRINT_NONNULL(logits, "logits");
    SPRINT_NONNULL(labels, "labels");
    SPRINT_NONNULL(loss, "loss");
    SPRINT_NONNULL(dlogits, "dlogits");
    SPRINT_ALIGNED(logits, "logits");
    SPRINT_ALIGNED(labels, "labels");
    SPRINT_ALIGNED(loss, "loss");
    SPRINT_ALIGNED(dlogits, "dlogits");
    return launch_xent(&logits, &labels, &loss, &dlogits, 1, N, C, reduction_sum, static_cast<cudaStream_t>(stream));
}

extern "C" int sprint_softmax_xent_batched(const float* const* logits, const int32_t* const* labels, float* const* loss,
                                           float* const* dlogits, int batch, int N, int C, int reduction_sum,
                                           sprint_stream_t stream) {
    SPRINT_REQUIRE(batch >= 0 && N >= 1 && C >= 1, SPRINT_ERR_SHAPE,
                   "%s: need batch >= 0, N >= 1 and C >= 1 (got %d, %d, %d)", __func__, batch, N, C);
    if (batch == 0) return SPRINT_OK;
    SPRINT_REQUIRE(logits && labels && loss && dlogits, SPRINT_ERR_INVALID_ARG, "%s: NULL pointer array", __func__);
    for (int g = 0; g < batch; ++g) {
        SPRINT_REQUIRE(logits[g] && labels[g] && loss[g] && dlogits[g], SPRINT_ERR_INVALID_ARG,
                       "%s: NULL pointer for problem %d", __func__, g);
        SPRINT_REQUIRE(aligned16(logits[g]) && aligned16(labels[g]) && aligned16(loss[g]) && aligned16(dlogits[g]),
                       SPRINT_ERR_ALIGN, "%s: pointer of problem %d not 16-byte aligned", __func__, g);
    }
    return launch_xent(logits, labels, loss, dlogits, batch, N, C, reduction_sum, static_cast<cudaStream_t>(stream));
}

extern "C" int sprint_im2col(const float* x, int N, int H, int W, int C, int pad, float* col, int32_t* src_index,
                             sprint_stream_t stream) {
    SPRINT_REQUIRE(N >= 1 && C >= 1 && (pad == 0 || pad == 1) && H + 2 * pad >= 3 && W + 2 * pad >= 3, SPRINT_ERR_SHAPE,
                   "%s: bad shape N=%d H=%d W=%d C=%d pad=%d", __func__, N, H, W, C, pad);
    const long long total = static_cast<long long>(N) * (H + 2 * pad - 2) * (W + 2 * pad - 2) * 9 * C;
    SPRINT_REQUIRE(total < (1ll << 31), SPRINT_ERR_SHAPE, "%s: output has %lld >= 2^31 elements", __func__, total);
    SPRINT_NONNULL(x, "x");
    SPRINT_NONNULL(col, "col");
    SPRINT_ALIGNED(x, "x");
    SPRINT_ALIGNED(col, "col");
    SPRINT_ALIGNED(src_index, "src_index");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (C % 4 == 0)
        im2col_kernel<4><<<grid_for(total / 4), 256, 0, s>>>(x, N, H, W, C, pad, col, src_index);
    else
        im2col_kernel<1><<<grid_for(total), 256, 0, s>>>(x, N, H, W, C, pad, col, src_index);
    return check_launch(__func__);
}

extern "C" int sprint_transpose(const float* src, float* dst, int rows, int cols, sprint_stream_t stream) {
    SPRINT_REQUIRE(rows >= 0 && cols >= 0, SPRINT_ERR_SHAPE, "%s: negative size", __func__);
    if (rows == 0 || cols == 0) return SPRINT_OK;
    SPRINT_NONNULL(src, "src");
    SPRINT_NONNULL(dst, "dst");
    SPRINT_REQUIRE(src != dst, SPRINT_ERR_INVALID_ARG, "%s: src and dst must not alias", __func__);
    return launch_transpose(src, dst, 1, rows, cols, 0, cols, 0, rows, static_cast<cudaStream_t>(stream));
}
