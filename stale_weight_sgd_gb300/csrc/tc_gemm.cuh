// tcgen05 TF32 GEMM engine for the contractions of the worker step.
//
// One CTA computes a 128 x BN tile of D = sum_k A(m,k) * B(n,k) over a range
// of 32-wide k-tiles (split-K over blockIdx.z where asked):
//   warp 4   : TMA producer (one lane) — fills a STAGES-deep ring of shared-
//              memory stages, 128 B (32 fp32) wide along k, 128-byte swizzled;
//   warp 5   : allocates the TMEM accumulator (BN fp32 columns x 128 lanes)
//              and issues tcgen05.mma.kind::tf32 (M=128, N=BN, K=8) from one
//              lane; tcgen05.commit frees a stage once its MMAs are done;
//   warps 0-3: epilogue — tcgen05.ld the accumulator (warp w owns TMEM lanes
//              32w..32w+31 = tile rows), apply bias/ReLU, the ReLU mask of the
//              backward pass, or the GradBuf accumulate, and store.
// Both operands are K-major (k contiguous in shared memory): the TF32 kind of
// tcgen05.mma reads no MN-major operand on this part, so transposed operands
// are formed in global memory by the callers (tc dispatch in gemm.cu).
// Every wait is bounded: one that gives up sets a bit in the device status
// word and the CTA runs to completion without hanging.
//
// Roles (the SGEMM roles of the SPRINT report, Sec. 3.3):
//   GEMM_2D   : A [M][K], B [N][K] row-major (fc, dedx fc with B = w^T,
//               dedw fc with A = dy^T and B = x^T)
//   CONV_IMPL : implicit-GEMM convolution — A = 128 NHWC pixels (4-D box,
//               shifted by the tap, halo zero-filled by TMA), B = the tap's
//               weight slice (3-D box). Forward: A = x, B = w[co][tap][ci];
//               dedx conv: A = dy at the mirrored tap, B = w^T[tap][ci][co].
//   CONV_WGRAD: dedw conv, per tap: A = dy^T [Cout][H][W][N], B = x^T
//               [Cin][H][W][N] shifted by the tap; a k-tile is 32 consecutive
//               (w, n) positions of one row (every TMA box here is 128 B wide
//               along its inner dimension, the 128-byte swizzle span).
#pragma once

#include "common.cuh"

namespace sprint {

enum Role : int { ROLE_GEMM_2D = 0, ROLE_CONV_IMPL = 1, ROLE_CONV_WGRAD = 2 };
enum Epi : int { EPI_STORE = 0, EPI_MASK = 1, EPI_ACCUM = 2 };

constexpr int TC_BM = 128;
constexpr int TC_BK = 32;                      // fp32 elements per 128-byte swizzle row
constexpr int TC_THREADS = 192;
constexpr int TC_A_STAGE = TC_BM * TC_BK * 4;  // 16 KB

__host__ __device__ constexpr int tc_stages(int bn) { return bn >= 256 ? 4 : (bn >= 128 ? 6 : 8); }
__host__ __device__ constexpr int tc_b_stage(int bn) { return bn * TC_BK * 4; }
__host__ __device__ constexpr int tc_tmem_cols(int bn) { return bn <= 32 ? 32 : (bn <= 64 ? 64 : (bn <= 128 ? 128 : 256)); }
__host__ __device__ constexpr int tc_smem_bytes(int bn) {
    return 1024 /* alignment slack */ + tc_stages(bn) * (TC_A_STAGE + tc_b_stage(bn)) + 256 /* barriers */;
}

struct TcParams {
    int M, N;            // GEMM_2D / CONV_WGRAD: output rows, columns; CONV_IMPL: N = columns
    int num_kt;          // k-tiles in the full reduction
    int kt_per_split;    // k-tiles per split
    int splits;          // CONV_WGRAD: blockIdx.z = tap * splits + split
    // convolution geometry: pixel boxes (bw x bh x bimg) tile the output grid
    int img_n, out_h, out_w, pad;
    int bw, bh, bimg, tiles_w, tiles_h;
    int chunks;          // CONV_IMPL: 32-channel chunks per tap
    int tap_sign;        // CONV_IMPL: +1 forward (x[p + tap - pad]), -1 dedx (dy[p - tap + pad])
    int b_tap_outer;     // CONV_IMPL: B map dims {k, n, 9} (1) or {k, 9, n} (0)
    // epilogue
    int epi;
    float* D;
    long long ldd;
    const float* bias;   // [N] or null
    const float* mask;   // ReLU mask source with D's layout, or null
    long long ldm;
    float alpha;
    int accumulate;
    int relu;
    float* partial;      // split-K partial sums [z][M][N] or null
    int* status;
};

#if defined(__CUDACC__)

template <int ROLE, int BN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcParams p) {
    constexpr int STAGES = tc_stages(BN);
    constexpr int B_STAGE = tc_b_stage(BN);
    constexpr uint32_t IDESC = idesc_tf32(BN, false, false);
    constexpr uint32_t TMEM_COLS = tc_tmem_cols(BN);
    constexpr uint32_t STAGE_BYTES = TC_A_STAGE + B_STAGE;
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN must be a multiple of 32 in [32, 256]");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * TC_A_STAGE;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_STAGE);
    uint64_t* empty = full + STAGES;
    uint64_t* accum_full = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_full + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    int split = blockIdx.z, tap = 0;
    if constexpr (ROLE == ROLE_CONV_WGRAD) {
        tap = blockIdx.z / p.splits;
        split = blockIdx.z % p.splits;
    }
    const int kt_begin = split * p.kt_per_split;
    int kt_end = kt_begin + p.kt_per_split;
    if (kt_end > p.num_kt) kt_end = p.num_kt;
    const int nkt = kt_end > kt_begin ? kt_end - kt_begin : 0;
    const int n0 = blockIdx.y * BN;
    const int m0 = blockIdx.x * TC_BM;

    // CONV_IMPL: the 128 output pixels of this tile
    int pw0 = 0, ph0 = 0, pn0 = 0;
    if constexpr (ROLE == ROLE_CONV_IMPL) {
        const int mt = blockIdx.x;
        pw0 = (mt % p.tiles_w) * p.bw;
        ph0 = ((mt / p.tiles_w) % p.tiles_h) * p.bh;
        pn0 = (mt / (p.tiles_w * p.tiles_h)) * p.bimg;
    }

    if (warp == 4 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum_full, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;

    if (warp == 4) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            for (int i = 0; i < nkt; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                if (!mbar_wait_bounded(&empty[s], ph ^ 1, p.status, DEV_FLAG_WAIT_PRODUCER)) break;
                const int kt = kt_begin + i;
                uint8_t* a_dst = sA + s * TC_A_STAGE;
                uint8_t* b_dst = sB + s * B_STAGE;
                mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                if constexpr (ROLE == ROLE_GEMM_2D) {
                    tma_load_2d(a_dst, &tmA, kt * TC_BK, m0, &full[s]);
                    tma_load_2d(b_dst, &tmB, kt * TC_BK, n0, &full[s]);
                } else if constexpr (ROLE == ROLE_CONV_IMPL) {
                    const int t = kt / p.chunks;
                    const int c0 = (kt % p.chunks) * TC_BK;
                    const int dh = (t / 3 - p.pad) * p.tap_sign, dw = (t % 3 - p.pad) * p.tap_sign;
                    tma_load_4d(a_dst, &tmA, c0, pw0 + dw, ph0 + dh, pn0, &full[s]);
                    if (p.b_tap_outer)
                        tma_load_3d(b_dst, &tmB, c0, n0, t, &full[s]);
                    else
                        tma_load_3d(b_dst, &tmB, c0, t, n0, &full[s]);
                } else {  // CONV_WGRAD: k-tile = 32 consecutive (w, n) of one output row h
                    // dy^T viewed as {Wo*N, Ho, Cout}, x^T as {W*N, H, Cin}: a tap shifts x by
                    // (kw - pad)*N along the inner dimension and by kh - pad rows; positions
                    // outside the image fall outside the tensor and are zero-filled.
                    const int h = kt / p.tiles_w;
                    const int c0 = (kt % p.tiles_w) * TC_BK;
                    tma_load_3d(a_dst, &tmA, c0, h, m0, &full[s]);
                    tma_load_3d(b_dst, &tmB, c0 + (tap % 3 - p.pad) * p.img_n, h + tap / 3 - p.pad, n0, &full[s]);
                }
            }
        }
    } else if (warp == 5) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            for (int i = 0; i < nkt; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                if (!mbar_wait_bounded(&full[s], ph, p.status, DEV_FLAG_WAIT_MMA)) break;
                tc_fence_after();
                const uint32_t a_base = smem_u32(sA + s * TC_A_STAGE);
                const uint32_t b_base = smem_u32(sB + s * B_STAGE);
#pragma unroll
                for (int kk = 0; kk < TC_BK / 8; ++kk) {
                    // K-major, 128-byte swizzle: 8 rows of 128 B per 1024-byte group (SBO);
                    // each K=8 step advances 32 bytes inside the swizzled row.
                    const uint64_t da = smem_desc_sw128(a_base + kk * 32, 16, 1024);
                    const uint64_t db = smem_desc_sw128(b_base + kk * 32, 16, 1024);
                    mma_tf32(tmem_d, da, db, IDESC, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
            }
            mma_commit(accum_full);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue (warps 0-3)
        const bool ok = mbar_wait_bounded(accum_full, 0, p.status, DEV_FLAG_WAIT_EPILOGUE);
        tc_fence_after();
        const int r = warp * 32 + lane;  // tile row = TMEM lane
        long long row_off = -1, mask_off = -1, part_off = -1;
        if constexpr (ROLE == ROLE_CONV_IMPL) {
            const int ow = pw0 + r % p.bw;
            const int oh = ph0 + (r / p.bw) % p.bh;
            const int on = pn0 + r / (p.bw * p.bh);
            if (ow < p.out_w && oh < p.out_h && on < p.img_n) {
                const long long pix = (static_cast<long long>(on) * p.out_h + oh) * p.out_w + ow;
                row_off = pix * p.ldd;
                mask_off = pix * p.ldm;
            }
        } else {
            const int m = m0 + r;
            if (m < p.M) {
                row_off = static_cast<long long>(m) * p.ldd;
                mask_off = static_cast<long long>(m) * p.ldm;
                if (p.partial) part_off = (static_cast<long long>(blockIdx.z) * p.M + m) * p.N;
            }
        }
        long long col_shift = 0;
        if constexpr (ROLE == ROLE_CONV_WGRAD) col_shift = static_cast<long long>(tap) * p.N;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem_d + (static_cast<uint32_t>(warp * 32) << 16) + c, v);
            tmem_wait_ld();
            const int ncol0 = n0 + c;
            if (!ok || row_off < 0 || nkt == 0 || ncol0 >= p.N) continue;
            const bool full4 = (ncol0 + 32 <= p.N);
            if (part_off >= 0) {
                float* dst = p.partial + part_off + ncol0;
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    if (full4) {
                        *reinterpret_cast<float4*>(dst + j) = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                                          __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (ncol0 + j + q < p.N) dst[j + q] = __uint_as_float(v[j + q]);
                    }
                }
                continue;
            }
            float* dst = p.D + row_off + col_shift + ncol0;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                float o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) o[q] = __uint_as_float(v[j + q]);
                if (p.epi == EPI_STORE) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float t = o[q];
                        if (p.bias && ncol0 + j + q < p.N) t += p.bias[ncol0 + j + q];
                        if (p.relu) t = fmaxf(t, 0.f);
                        o[q] = t;
                    }
                } else if (p.epi == EPI_MASK) {
                    if (p.mask) {
                        const float* ms = p.mask + mask_off + ncol0 + j;
                        if (full4) {
                            const float4 mv = *reinterpret_cast<const float4*>(ms);
                            o[0] = mv.x > 0.f ? o[0] : 0.f;
                            o[1] = mv.y > 0.f ? o[1] : 0.f;
                            o[2] = mv.z > 0.f ? o[2] : 0.f;
                            o[3] = mv.w > 0.f ? o[3] : 0.f;
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (ncol0 + j + q < p.N) o[q] = ms[q] > 0.f ? o[q] : 0.f;
                        }
                    }
                } else {  // EPI_ACCUM: GradBuf <- (accumulate ? GradBuf : 0) + alpha * acc
                    if (full4) {
                        float4 prev = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (p.accumulate) prev = *reinterpret_cast<const float4*>(dst + j);
                        o[0] = prev.x + p.alpha * o[0];
                        o[1] = prev.y + p.alpha * o[1];
                        o[2] = prev.z + p.alpha * o[2];
                        o[3] = prev.w + p.alpha * o[3];
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (ncol0 + j + q < p.N) o[q] = (p.accumulate ? dst[j + q] : 0.f) + p.alpha * o[q];
                    }
                }
                if (full4) {
                    *reinterpret_cast<float4*>(dst + j) = make_float4(o[0], o[1], o[2], o[3]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (ncol0 + j + q < p.N) dst[j + q] = o[q];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem_d, TMEM_COLS);
    }
}

#endif  // __CUDACC__

}  // namespace sprint
