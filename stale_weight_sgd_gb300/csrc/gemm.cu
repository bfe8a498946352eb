// FC and convolution entry points of libsprint: tile/box/split selection,
// TMA tensor maps, launches of the tcgen05 engine (tc_gemm.cuh), split-K
// reduction, and CUDA-core kernels for shapes the tensor-core loaders cannot
// tile (channel counts that are not multiples of 32, e.g. the RGB input
// layer; FC widths that are not multiples of 4, e.g. a 10-way classifier).
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "tc_gemm.cuh"
#include "tc_halo.cuh"

namespace sprint {

int launch_colsum(const float* in, long long rows, int cols, float* partial, float* out, float alpha, int accumulate,
                  cudaStream_t s);
int colsum_chunks(long long rows, int cols);
int launch_transpose(const float* src, float* dst, int batch, int R, int C, long long sb, long long sr, long long db,
                     long long dc, cudaStream_t s, long long drt = 32);
int launch_transpose_group(const float* const* src, float* const* dst, int G, int R, int C, cudaStream_t s);
int launch_transpose_colsum(const float* src, float* dst, int batch, int R, int C, long long sb, long long sr,
                            long long db, long long dc, float* partial, float* out, float alpha, int accumulate,
                            cudaStream_t s, long long drt = 32);
int launch_colsum_group(const float* const* in, float* const* out, int G, long long rows, int cols, float alpha,
                        int accumulate, cudaStream_t s);

namespace {

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// fp32 tensor map, 128-byte swizzle, zero fill out of bounds. dims[0] is the
// contiguous dimension; strides are in bytes for dims 1..rank-1. The TFLOAT32
// element type makes the copy round each fp32 value to TF32 (to nearest) on
// its way into shared memory, so the tensor core sees round-to-nearest
// operands instead of truncating the low mantissa bits itself (measured: 3.6x
// smaller median relative error of the products, no systematic bias).
bool make_tmap(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
               const uint32_t* box, bool tf32_load = true) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i + 1 < rank; ++i) gs[i] = strides[i];
    // loads: TFLOAT32 (round to nearest on the way in); stores: FLOAT32 (bit-exact)
    CUresult r = fn(m, tf32_load ? CU_TENSOR_MAP_DATA_TYPE_TFLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank,
                    const_cast<void*>(base), gd, gs, bx, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ tcgen05 launches
// Tile shape of one launch: BN output columns per tile; pair = clusters of two
// CTAs sharing M = 256 MMAs (each CTA loads BN/2 rows of B).
struct Tile {
    int bn = 64;
    bool pair = false;
    uint32_t b_rows() const { return static_cast<uint32_t>(pair ? bn / 2 : bn); }
};

// CTA pairs that can be resident at once for this kernel (clusters are placed
// within one GPC, so this can be below half the SM count)
template <int ROLE, int BN, int G>
int pair_slots() {
    static int slots[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!slots[dev]) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
        cfg.blockDim = dim3(tc_threads<ROLE>(), 1, 1);
        cfg.dynamicSmemBytes = tc_smem_bytes_r<ROLE>(BN, true);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<ROLE, BN, true, G>, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = num_sms() / 2;
        }
        slots[dev] = n;
    }
    return slots[dev];
}

template <int ROLE, int BN, bool PAIR, int G>
int launch_tc_bn(const TcMaps<G>& maps, const TcParams& p, cudaStream_t s) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(tc_gemm_kernel<ROLE, BN, PAIR, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tc_smem_bytes_r<ROLE>(BN, PAIR)) != cudaSuccess)
            return check_cuda("cudaFuncSetAttribute(tc_gemm_kernel)");
        attr_done[dev] = true;
    }
    const int work = p.num_tiles;
    if constexpr (!PAIR) {
        // persistent: one CTA per SM at most, each walking tiles blockIdx.x, +gridDim.x, ...
        const int grid = work < num_sms() ? work : num_sms();
        tc_gemm_kernel<ROLE, BN, false, G><<<grid, tc_threads<ROLE>(), tc_smem_bytes_r<ROLE>(BN, false), s>>>(maps, p);
        return check_launch("tc_gemm_kernel");
    } else {
        // persistent pairs: at most as many clusters as can be resident together
        const int slots = pair_slots<ROLE, BN, G>();
        const int pairs = work < slots ? work : slots;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * pairs, 1, 1);
        cfg.blockDim = dim3(tc_threads<ROLE>(), 1, 1);
        cfg.dynamicSmemBytes = tc_smem_bytes_r<ROLE>(BN, true);
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaLaunchKernelEx(&cfg, tc_gemm_kernel<ROLE, BN, true, G>, maps, p);
        return check_launch("tc_gemm_kernel(pair)");
    }
}

// m_tiles counts 128-row tiles; a pair launch walks ceil(m_tiles / 2) units.
// For a grouped launch (G > 1) z_tiles is the number of problems.
template <int ROLE, int G>
int launch_tc_maps(Tile tl, const TcMaps<G>& maps, TcParams p, long long m_tiles, long long n_tiles,
                   long long z_tiles, cudaStream_t s) {
    const long long m_units = tl.pair ? (m_tiles + 1) / 2 : m_tiles;
    long long tiles = m_units * n_tiles * z_tiles;
    if (tiles <= 0) return SPRINT_OK;
    if (p.tail_splits > 1) tiles = p.tail_start + (tiles - p.tail_start) * p.tail_splits;
    if (tiles > (1ll << 31) - 1) return fail(SPRINT_ERR_SHAPE, "tc_gemm: %lld tiles is too many", tiles);
    p.m_tiles = static_cast<int>(m_units);
    p.n_tiles = static_cast<int>(n_tiles);
    p.z_tiles = static_cast<int>(z_tiles);
    p.num_tiles = static_cast<int>(tiles);
    if (tl.pair) {
        switch (tl.bn) {
            case 64: return launch_tc_bn<ROLE, 64, true, G>(maps, p, s);
            case 128: return launch_tc_bn<ROLE, 128, true, G>(maps, p, s);
            case 160: return launch_tc_bn<ROLE, 160, true, G>(maps, p, s);
            case 192: return launch_tc_bn<ROLE, 192, true, G>(maps, p, s);
            case 256: return launch_tc_bn<ROLE, 256, true, G>(maps, p, s);
            default: return fail(SPRINT_ERR_UNSUPPORTED, "tile width %d not built", tl.bn);
        }
    }
    switch (tl.bn) {
        case 64: return launch_tc_bn<ROLE, 64, false, G>(maps, p, s);
        case 128: return launch_tc_bn<ROLE, 128, false, G>(maps, p, s);
        case 160: return launch_tc_bn<ROLE, 160, false, G>(maps, p, s);
        case 192: return launch_tc_bn<ROLE, 192, false, G>(maps, p, s);
        case 256: return launch_tc_bn<ROLE, 256, false, G>(maps, p, s);
        default: return fail(SPRINT_ERR_UNSUPPORTED, "tile width %d not built", tl.bn);
    }
}

template <int ROLE>
int launch_tc(Tile tl, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d, TcParams p,
              long long m_tiles, long long n_tiles, long long z_tiles, cudaStream_t s) {
    TcMaps<1> maps;
    maps.a[0] = a;
    maps.b[0] = b;
    maps.d[0] = d;
    return launch_tc_maps<ROLE, 1>(tl, maps, p, m_tiles, n_tiles, z_tiles, s);
}

// Picks the tile shape of a persistent launch. Each slot (an SM, or a pair of
// SMs) runs ceil(units / slots) work units one after another; a unit's time
// grows with its width and shrinks with the MMA efficiency of that shape, so
// minimise ceil(units / slots) * bn / efficiency. A pair unit is two 128-row
// tiles on two SMs, so it takes as long as one single-CTA tile of the same
// width at the same efficiency. The efficiencies are measured (8192^3 TF32
// GEMM, relative to the pair of width 256 at ~940 TFLOP/s): a TF32 k-tile is
// bound by shared-memory bandwidth (the TMA writes plus the tensor core's
// operand reads, ~128 B/clk per SM), which only the pair-256 shape, loading half
// of B per SM and reading A once per 256 columns, brings under its MMA time.
Tile pick_tile(long long m_tiles, long long n, long long z, int max_bn) {
    const int cands[5] = {256, 192, 160, 128, 64};
    const double eff[5] = {0.86, 0.72, 0.68, 0.58, 0.36};
    const double eff_pair[5] = {1.0, 0.79, 0.86, 0.74, 0.40};
    const long long sms = num_sms();
    Tile best;
    double best_cost = 1e300;
    for (int pair = 0; pair < 2; ++pair) {
        if (pair && m_tiles < 2) continue;
        const long long mu = pair ? (m_tiles + 1) / 2 : m_tiles;
        const long long slots = pair ? sms / 2 : sms;
        for (int i = 0; i < 5; ++i) {
            const int bn = cands[i];
            if (bn > max_bn) continue;
            const long long units = mu * ((n + bn - 1) / bn) * z;
            const long long rounds = (units + slots - 1) / slots;
            const double cost = static_cast<double>(rounds) * bn / (pair ? eff_pair[i] : eff[i]);
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best.bn = bn;
                best.pair = pair != 0;
            }
        }
    }
    return best;
}

// Shared memory slabs the tail split may use: at most one TM x BN slab per
// slot of the last round (TM x slots = 128 x SMs rows, BN <= 256).
size_t tail_bytes() { return static_cast<size_t>(num_sms()) * TC_BM * 256 * 4; }

// A launch plan: tile shape, plus the k-split of the last, partial round's
// tiles (tail_splits == 1: none). With the split the last round runs r * s
// units of 1/s of the k range on the slots the r leftover tiles would leave
// idle; the slabs are added afterwards (tc_tail_reduce).
struct GemmPlan {
    Tile tile;
    int tail_splits = 1, tail_kt = 0;
    long long tail_start = 0;
};

GemmPlan plan_gemm(long long m_tiles, long long n, long long z, int max_bn, int num_kt, bool allow_tail) {
    const int cands[5] = {256, 192, 160, 128, 64};
    const double eff[5] = {0.86, 0.72, 0.68, 0.58, 0.36};
    const double eff_pair[5] = {1.0, 0.79, 0.86, 0.74, 0.40};
    const long long sms = num_sms();
    GemmPlan best;
    double best_cost = 1e300;
    for (int pair = 0; pair < 2; ++pair) {
        if (pair && m_tiles < 2) continue;
        const long long mu = pair ? (m_tiles + 1) / 2 : m_tiles;
        const long long slots = pair ? sms / 2 : sms;
        for (int i = 0; i < 5; ++i) {
            const int bn = cands[i];
            if (bn > max_bn) continue;
            const long long units = mu * ((n + bn - 1) / bn) * z;
            const long long full = units / slots, r = units % slots;
            double rounds = static_cast<double>(full);
            long long sp = 1;
            if (r > 0) {
                // the last round whole, or cut into s k-ranges plus the slab reduction, whose
                // time (measured: ~4 us plus its slabs' traffic at ~4 TB/s) is counted in units
                // of one unit's MMA time (~0.34 us per k-tile of a 256 x 256 pair tile at full
                // rate, scaled by width / efficiency like the cost below)
                const double e = pair ? eff_pair[i] : eff[i];
                const double unit_us = static_cast<double>(num_kt) * 0.34 * (bn / 256.0) / e;
                const double tile_bytes = (pair ? 256.0 : 128.0) * bn * 4.0;
                double best_tail = 1.0;
                long long smax = allow_tail ? slots / r : 1;
                if (smax > num_kt / 4) smax = num_kt / 4;
                for (long long c = 2; c <= smax; ++c) {
                    // equal k-ranges of ceil(num_kt / c) k-tiles: no range may be empty
                    const long long kt = (num_kt + c - 1) / c;
                    const long long cs = (num_kt + kt - 1) / kt;
                    if (cs < 2) continue;
                    const double reduce_us = 4.0 + static_cast<double>(r) * cs * tile_bytes / 4e6;
                    const double tail = 1.0 / static_cast<double>(cs) + reduce_us / unit_us;
                    if (tail < best_tail - 1e-9) {
                        best_tail = tail;
                        sp = cs;
                    }
                }
                rounds += best_tail;
            }
            const double cost = rounds * bn / (pair ? eff_pair[i] : eff[i]);
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best.tile.bn = bn;
                best.tile.pair = pair != 0;
                best.tail_splits = static_cast<int>(sp);
                best.tail_kt = sp > 1 ? static_cast<int>((num_kt + sp - 1) / sp) : 0;
                best.tail_start = full * slots;
            }
        }
    }
    return best;
}

// Launches tc_tail_reduce for the tail tiles of a GEMM_2D launch planned by
// plan_gemm; m_units / n_tiles / z_tiles describe that launch's unit grid
// (the kernel decomposes tile indices with them).
template <int ROLE>
int launch_tail_reduce(const GemmPlan& pl, TcParams p, long long m_units, long long n_tiles, long long z_tiles,
                       cudaStream_t s) {
    p.m_tiles = static_cast<int>(m_units);
    p.n_tiles = static_cast<int>(n_tiles);
    p.z_tiles = static_cast<int>(z_tiles);
    const long long total_units = m_units * n_tiles * z_tiles;
    if (p.m_tiles <= 0 || p.n_tiles <= 0 || total_units <= pl.tail_start) return SPRINT_OK;
    const int tiles = static_cast<int>(total_units - pl.tail_start);
    const long long work = static_cast<long long>(tiles) * (pl.tile.pair ? 256 : 128) * (pl.tile.bn / 4);
    long long blocks = (work + 255) / 256;
    if (blocks > 8ll * num_sms()) blocks = 8ll * num_sms();
    const unsigned g = static_cast<unsigned>(blocks);
#define SPRINT_TAIL(BNV)                                                              \
    case BNV:                                                                         \
        if (pl.tile.pair)                                                             \
            tc_tail_reduce<BNV, 256, ROLE><<<g, 256, 0, s>>>(p, tiles);               \
        else                                                                          \
            tc_tail_reduce<BNV, 128, ROLE><<<g, 256, 0, s>>>(p, tiles);               \
        break;
    switch (pl.tile.bn) {
        SPRINT_TAIL(64)
        SPRINT_TAIL(128)
        SPRINT_TAIL(160)
        SPRINT_TAIL(192)
        SPRINT_TAIL(256)
        default: return fail(SPRINT_ERR_UNSUPPORTED, "tile width %d not built", pl.tile.bn);
    }
#undef SPRINT_TAIL
    return check_launch("tc_tail_reduce");
}

TcParams base_params() {
    TcParams p;
    memset(&p, 0, sizeof(p));
    p.alpha = 1.f;
    p.splits = 1;
    p.tap_sign = 1;
    p.vec_col = -1;
    p.status = device_status_ptr();
    return p;
}

// A box of `pixels` output pixels (bw x bh x bimg, powers of two) that covers
// the grid w x h x n with the fewest boxes.
struct PixBox {
    int bw, bh, bimg, tw, th, tn;
    long long tiles() const { return static_cast<long long>(tw) * th * tn; }
};

PixBox pick_box(int pixels, int w, int h, int n, int min_bimg = 1) {
    PixBox best{0, 0, 0, 0, 0, 0};
    long long best_tiles = -1;
    for (int bw = 1; bw <= pixels && bw <= 256; bw *= 2)
        for (int bh = 1; bw * bh <= pixels && bh <= 256; bh *= 2) {
            const int bimg = pixels / (bw * bh);
            if (bimg > 256 || bimg < min_bimg || bw * bh * bimg != pixels) continue;
            PixBox b{bw, bh, bimg, (w + bw - 1) / bw, (h + bh - 1) / bh, (n + bimg - 1) / bimg};
            const long long t = b.tiles();
            // fewest boxes; on a tie prefer the widest rows (longest contiguous runs)
            if (best_tiles < 0 || t < best_tiles || (t == best_tiles && bw > best.bw)) {
                best = b;
                best_tiles = t;
            }
        }
    return best;
}

// ------------------------------------------------------------------ CUDA-core kernels
enum SimtEpi : int { SIMT_STORE = 0, SIMT_MASK = 1, SIMT_ACCUM = 2 };

struct SimtGemm {
    int M, N, K;
    const float* A;
    long long a_sm, a_sk;
    const float* B;
    long long b_sn, b_sk;
    float* D;
    long long ldd;
    const float* bias;
    const float* mask;
    long long ldm;
    float alpha;
    int accumulate, relu, epi;
};

// D[m][n] = epi(sum_k A[m*a_sm + k*a_sk] * B[n*b_sn + k*b_sk]); 64x64 tile, 4x4 per thread.
__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtGemm g) {
    __shared__ float As[16][64 + 1];
    __shared__ float Bs[16][64 + 1];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < g.K; k0 += 16) {
        // consecutive threads walk the operand's contiguous dimension (k when
        // its k-stride is 1, else m / n), so the loads coalesce
        for (int e = threadIdx.x; e < 16 * 64; e += 256) {
            const int kk = g.a_sk == 1 ? e % 16 : e / 64, mm = g.a_sk == 1 ? e / 16 : e % 64;
            const int m = m0 + mm, k = k0 + kk;
            As[kk][mm] = (m < g.M && k < g.K) ? g.A[m * g.a_sm + k * g.a_sk] : 0.f;
        }
        for (int e = threadIdx.x; e < 16 * 64; e += 256) {
            const int kk = g.b_sk == 1 ? e % 16 : e / 64, nn = g.b_sk == 1 ? e / 16 : e % 64;
            const int n = n0 + nn, k = k0 + kk;
            Bs[kk][nn] = (n < g.N && k < g.K) ? g.B[n * g.b_sn + k * g.b_sk] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[kk][ty * 4 + i];
                b[i] = Bs[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= g.M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= g.N) continue;
            float v = acc[i][j];
            float* d = g.D + m * g.ldd + n;
            if (g.epi == SIMT_STORE) {
                if (g.bias) v += g.bias[n];
                if (g.relu) v = fmaxf(v, 0.f);
            } else if (g.epi == SIMT_MASK) {
                if (g.mask && !(g.mask[m * g.ldm + n] > 0.f)) v = 0.f;
            } else {
                v = (g.accumulate ? *d : 0.f) + g.alpha * v;
            }
            *d = v;
        }
    }
}

int launch_simt_gemm(const SimtGemm& g, cudaStream_t s) {
    dim3 grid((g.N + 63) / 64, (g.M + 63) / 64);
    simt_gemm_kernel<<<grid, 256, 0, s>>>(g);
    return check_launch("simt_gemm_kernel");
}

// Skinny product for few output columns (N <= 16), both operands k-contiguous:
// D[m][n] = act(bias[n] + sum_k A[m*lda + k] * B[n*ldb + k]). Two rows per
// block; the 256 threads split k, keep every partial sum in registers, and
// reduce in a fixed order (warp shuffles, then the 8 warps in order).
constexpr int kSkinnyN = 16;
__global__ void __launch_bounds__(256) skinny_nt_kernel(const float* __restrict__ A, long long lda,
                                                        const float* __restrict__ B, long long ldb,
                                                        const float* __restrict__ bias, float* __restrict__ D,
                                                        long long ldd, int M, int N, int K, int relu) {
    __shared__ float red[8][2][kSkinnyN];
    const int m0 = blockIdx.x * 2;
    const bool two = m0 + 1 < M;
    const float* a0 = A + static_cast<long long>(m0) * lda;
    const float* a1 = A + static_cast<long long>(two ? m0 + 1 : m0) * lda;
    float acc0[kSkinnyN], acc1[kSkinnyN];
#pragma unroll
    for (int n = 0; n < kSkinnyN; ++n) acc0[n] = acc1[n] = 0.f;
    for (int k = threadIdx.x; k < K; k += 256) {
        const float x0 = a0[k], x1 = a1[k];
#pragma unroll
        for (int n = 0; n < kSkinnyN; ++n) {
            if (n < N) {
                const float w = B[static_cast<long long>(n) * ldb + k];
                acc0[n] = fmaf(x0, w, acc0[n]);
                acc1[n] = fmaf(x1, w, acc1[n]);
            }
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int n = 0; n < kSkinnyN; ++n) {
        float u = acc0[n], v = acc1[n];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            u += __shfl_xor_sync(0xffffffffu, u, o);
            v += __shfl_xor_sync(0xffffffffu, v, o);
        }
        if (lane == 0) {
            red[warp][0][n] = u;
            red[warp][1][n] = v;
        }
    }
    __syncthreads();
    if (threadIdx.x < 2 * kSkinnyN) {
        const int r = threadIdx.x / kSkinnyN, n = threadIdx.x % kSkinnyN;
        if (n < N && (r == 0 || two)) {
            float t = red[0][r][n];
#pragma unroll
            for (int w = 1; w < 8; ++w) t += red[w][r][n];
            if (bias) t += bias[n];
            if (relu) t = fmaxf(t, 0.f);
            D[static_cast<long long>(m0 + r) * ldd + n] = t;
        }
    }
}

// im2col with the k dimension padded to kp (>= 9*C, a multiple of 32) with
// zeros: col[p][k] = x[n][oh+kh-pad][ow+kw-pad][ci] for k = (kh*3+kw)*C + ci < 9C.
// Used for input layers whose channel count TMA cannot tile (e.g. RGB).
__global__ void __launch_bounds__(256) im2col_pad_kernel(const float* __restrict__ x, int N, int H, int W, int C,
                                                         int pad, int kp, float* __restrict__ col) {
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    const long long total = static_cast<long long>(N) * Ho * Wo * kp;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int k = static_cast<int>(idx % kp);
        const long long pix = idx / kp;
        float v = 0.f;
        if (k < 9 * C) {
            const int ow = static_cast<int>(pix % Wo);
            const int oh = static_cast<int>((pix / Wo) % Ho);
            const long long n = pix / (static_cast<long long>(Wo) * Ho);
            const int tap = k / C, ci = k % C;
            const int ih = oh + tap / 3 - pad, iw = ow + tap % 3 - pad;
            if (ih >= 0 && ih < H && iw >= 0 && iw < W) v = x[((n * H + ih) * W + iw) * C + ci];
        }
        col[idx] = v;
    }
}

// wp[co][k] = w[co][k] for k < K, 0 for K <= k < kp
__global__ void pad_cols_kernel(const float* __restrict__ w, int rows, int K, int kp, float* __restrict__ wp) {
    const int total = rows * kp;
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
        const int k = idx % kp, r = idx / kp;
        wp[idx] = k < K ? w[r * K + k] : 0.f;
    }
}

// Narrow outputs (N <= 16, e.g. a 10-way classifier), K % 4 == 0, up to
// kMaxGroup problems per launch (blockIdx.y = problem): a block of 256 threads
// owns 4 rows of one problem; every thread walks k in float4 steps (stride
// 256 * 4) for the 4 rows and all N outputs, so each w float4 it loads serves 4
// rows; partial sums are reduced in a fixed order (warp shuffles, then the 8
// warps in order).
struct SkinnyGroup {
    const float* x[kMaxGroup];
    const float* w[kMaxGroup];
    const float* b[kMaxGroup];
    float* y[kMaxGroup];
};

template <int NO>
__global__ void __launch_bounds__(256) skinny4_kernel(SkinnyGroup grp, int M, int N, int K, int relu) {
    __shared__ float red[8][4][NO];
    const int g = blockIdx.y;
    const float* __restrict__ X = grp.x[g];
    const float* __restrict__ Wt = grp.w[g];
    const int m0 = blockIdx.x * 4;
    const int K4 = K >> 2;
    float acc[4][NO];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int n = 0; n < NO; ++n) acc[r][n] = 0.f;
    const float4* xr[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int m = m0 + r < M ? m0 + r : M - 1;   // rows past M repeat the last row (not stored)
        xr[r] = reinterpret_cast<const float4*>(X + static_cast<long long>(m) * K);
    }
    for (int k4 = threadIdx.x; k4 < K4; k4 += 256) {
        // every load of this k-step is issued before the first FMA uses one
        float4 xv[4], wv[NO];
#pragma unroll
        for (int r = 0; r < 4; ++r) xv[r] = __ldcs(xr[r] + k4);
#pragma unroll
        for (int n = 0; n < NO; ++n)
            wv[n] = n < N ? __ldg(reinterpret_cast<const float4*>(Wt + static_cast<long long>(n) * K) + k4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int n = 0; n < NO; ++n)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float a = acc[r][n];
                a = fmaf(xv[r].x, wv[n].x, a);
                a = fmaf(xv[r].y, wv[n].y, a);
                a = fmaf(xv[r].z, wv[n].z, a);
                a = fmaf(xv[r].w, wv[n].w, a);
                acc[r][n] = a;
            }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int n = 0; n < NO; ++n) {
            if (n < N) {
                float v = acc[r][n];
#pragma unroll
                for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) red[warp][r][n] = v;
            }
        }
    __syncthreads();
    if (threadIdx.x < 4 * NO) {
        const int r = threadIdx.x / NO, n = threadIdx.x % NO;
        if (n < N && m0 + r < M) {
            float t = red[0][r][n];
#pragma unroll
            for (int w = 1; w < 8; ++w) t += red[w][r][n];
            if (grp.b[g]) t += grp.b[g][n];
            if (relu) t = fmaxf(t, 0.f);
            grp.y[g][static_cast<long long>(m0 + r) * N + n] = t;
        }
    }
}

// y_g = x_g . w_g^T (+ b_g, ReLU) for narrow outputs (N <= 16, K % 4 == 0)
int launch_skinny4(const float* const* x, const float* const* w, const float* const* b, float* const* y, int G,
                   int M, int N, int K, int relu, cudaStream_t s) {
    for (int g0 = 0; g0 < G; g0 += kMaxGroup) {
        const int n = G - g0 < kMaxGroup ? G - g0 : kMaxGroup;
        SkinnyGroup t{};
        for (int i = 0; i < n; ++i) {
            t.x[i] = x[g0 + i];
            t.w[i] = w[g0 + i];
            t.b[i] = b ? b[g0 + i] : nullptr;
            t.y[i] = y[g0 + i];
        }
        const dim3 grid((M + 3) / 4, n);
        if (N <= 4)
            skinny4_kernel<4><<<grid, 256, 0, s>>>(t, M, N, K, relu);
        else if (N <= 8)
            skinny4_kernel<8><<<grid, 256, 0, s>>>(t, M, N, K, relu);
        else if (N <= 10)
            skinny4_kernel<10><<<grid, 256, 0, s>>>(t, M, N, K, relu);
        else
            skinny4_kernel<kSkinnyN><<<grid, 256, 0, s>>>(t, M, N, K, relu);
        const int rc = check_launch("skinny4_kernel");
        if (rc) return rc;
    }
    return SPRINT_OK;
}

// dx[m][n] = mask(m, n) * sum_{k < K} dy[m][k] * w[k][n] for a short reduction
// (K <= 32, e.g. the input gradient of a 10-way classifier): one thread per
// output, dy row broadcast within the warp, w read coalesced along n.
__global__ void __launch_bounds__(256) smallk_dx_kernel(const float* __restrict__ dy, const float* __restrict__ w,
                                                        const float* __restrict__ mask, float* __restrict__ dx, int M,
                                                        int N, int K) {
    const long long total = static_cast<long long>(M) * N;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(idx % N);
        const long long m = idx / N;
        if (mask && !(mask[idx] > 0.f)) {
            dx[idx] = 0.f;
            continue;
        }
        const float* d = dy + m * K;
        float acc = 0.f;
        for (int k = 0; k < K; ++k) acc = fmaf(d[k], w[static_cast<long long>(k) * N + n], acc);
        dx[idx] = acc;
    }
}

// Grouped form for N % 4 == 0 (blockIdx.y = problem): a thread computes 4
// consecutive outputs of one row from the row's K dy values (broadcast) and K
// float4 loads of w, all issued before the FMAs.
struct SmallkGroup {
    const float* dy[kMaxGroup];
    const float* w[kMaxGroup];
    const float* mask[kMaxGroup];
    float* dx[kMaxGroup];
    float* dxT[kMaxGroup];
};

// dx = mask * (dy . w) for a short reduction (K <= 32, e.g. the classifier's 10
// outputs), optionally with dxT = dx^T ([N][M]). A thread owns one float4 of
// columns for SK_ROWS consecutive rows: its K float4 of w are loaded once and
// reused for every row; a warp covers 128 consecutive columns (512-byte rows
// of dx, mask). dxT gets the thread's SK_ROWS-long column runs (32 bytes per
// column, two float4 when M % 4 == 0).
constexpr int SK_ROWS = 8;

template <int KM>
__global__ void __launch_bounds__(256) smallk_dx4_kernel(SmallkGroup grp, int M, int N, int K) {
    const int g = blockIdx.y;
    const float* __restrict__ dy = grp.dy[g];
    const float4* __restrict__ w4 = reinterpret_cast<const float4*>(grp.w[g]);
    const float* __restrict__ mask = grp.mask[g];
    float4* __restrict__ dx4 = reinterpret_cast<float4*>(grp.dx[g]);
    float* __restrict__ dxT = grp.dxT[g];
    const int N4 = N >> 2;
    const int row_blocks = (M + SK_ROWS - 1) / SK_ROWS;
    const long long total = static_cast<long long>(row_blocks) * N4;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int n4 = static_cast<int>(idx % N4);
        const int m0 = static_cast<int>(idx / N4) * SK_ROWS;
        float4 wv[KM];
#pragma unroll
        for (int k = 0; k < KM; ++k)
            wv[k] = k < K ? __ldg(w4 + static_cast<long long>(k) * N4 + n4) : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 out[SK_ROWS];
#pragma unroll
        for (int i = 0; i < SK_ROWS; ++i) {
            const int m = m0 + i;
            out[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m >= M) continue;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < KM; ++k) {
                if (k >= K) break;
                const float d = dy[static_cast<long long>(m) * K + k];
                a.x = fmaf(d, wv[k].x, a.x);
                a.y = fmaf(d, wv[k].y, a.y);
                a.z = fmaf(d, wv[k].z, a.z);
                a.w = fmaf(d, wv[k].w, a.w);
            }
            const long long e = static_cast<long long>(m) * N4 + n4;
            if (mask) {
                const float4 mk = __ldcs(reinterpret_cast<const float4*>(mask) + e);
                a.x = mk.x > 0.f ? a.x : 0.f;
                a.y = mk.y > 0.f ? a.y : 0.f;
                a.z = mk.z > 0.f ? a.z : 0.f;
                a.w = mk.w > 0.f ? a.w : 0.f;
            }
            __stcs(dx4 + e, a);
            out[i] = a;
        }
        if (dxT) {
            const int c = 4 * n4;
            const float col[4][SK_ROWS] = {
                {out[0].x, out[1].x, out[2].x, out[3].x, out[4].x, out[5].x, out[6].x, out[7].x},
                {out[0].y, out[1].y, out[2].y, out[3].y, out[4].y, out[5].y, out[6].y, out[7].y},
                {out[0].z, out[1].z, out[2].z, out[3].z, out[4].z, out[5].z, out[6].z, out[7].z},
                {out[0].w, out[1].w, out[2].w, out[3].w, out[4].w, out[5].w, out[6].w, out[7].w}};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float* dst = dxT + static_cast<long long>(c + q) * M + m0;
                if ((M & 3) == 0 && m0 + SK_ROWS <= M) {
                    __stcs(reinterpret_cast<float4*>(dst), make_float4(col[q][0], col[q][1], col[q][2], col[q][3]));
                    __stcs(reinterpret_cast<float4*>(dst + 4), make_float4(col[q][4], col[q][5], col[q][6], col[q][7]));
                } else {
#pragma unroll
                    for (int i = 0; i < SK_ROWS; ++i)
                        if (m0 + i < M) dst[i] = col[q][i];
                }
            }
        }
    }
}

// dx_g = mask_g * (dy_g . w_g) (and dxT_g = dx_g^T when dxT is given) for K <= 32,
// N % 4 == 0, all problems in as few launches as possible
int launch_smallk_dx4(const float* const* dy, const float* const* w, const float* const* mask, float* const* dx,
                      float* const* dxT, int G, int M, int N, int K, cudaStream_t s) {
    static_assert(SK_ROWS == 8, "the transposed store is written for 8-row runs");
    const long long total = static_cast<long long>((M + SK_ROWS - 1) / SK_ROWS) * (N / 4);
    long long blocks = (total + 255) / 256;
    const long long cap = 8ll * num_sms();
    if (blocks > cap) blocks = cap;
    for (int g0 = 0; g0 < G; g0 += kMaxGroup) {
        const int n = G - g0 < kMaxGroup ? G - g0 : kMaxGroup;
        SmallkGroup t{};
        for (int i = 0; i < n; ++i) {
            t.dy[i] = dy[g0 + i];
            t.w[i] = w[g0 + i];
            t.mask[i] = mask ? mask[g0 + i] : nullptr;
            t.dx[i] = dx[g0 + i];
            t.dxT[i] = dxT ? dxT[g0 + i] : nullptr;
        }
        const dim3 grid(static_cast<unsigned>(blocks), n);
        if (K <= 8)
            smallk_dx4_kernel<8><<<grid, 256, 0, s>>>(t, M, N, K);
        else if (K <= 16)
            smallk_dx4_kernel<16><<<grid, 256, 0, s>>>(t, M, N, K);
        else
            smallk_dx4_kernel<32><<<grid, 256, 0, s>>>(t, M, N, K);
        const int rc = check_launch("smallk_dx4_kernel");
        if (rc) return rc;
    }
    return SPRINT_OK;
}

// Forward convolution with very few input channels (the RGB layer, CIN <= 4,
// Cout % 16 == 0). Its 9*CIN-long reduction makes it bound by writing y, not by
// arithmetic (~14 FLOP per output byte), so it runs on the CUDA cores: a
// thread owns PX horizontally adjacent output pixels x 16 consecutive output
// channels, loads their shared 3 x (PX+2) x CIN input window once (zero
// outside the image), and reads the weights — staged per block in shared
// memory as [tap*CIN+ci][co] — as four float4 per tap, each used for all PX
// pixels; bias and ReLU are fused and y is written as float4. The 32 lanes of
// a warp take 32 consecutive pixel groups of the same channel group, so every
// weight read is a shared-memory broadcast (lanes of different groups in one
// warp read rows 64 B apart: bank conflicts, measured 10x slower). With one
// pixel per thread the weight reads kept the shared-memory pipe 89% busy (ncu)
// at ~1.3 TB/s of output; PX pixels per read divide them by PX. PX = 2:
// 0.58 -> 0.46 ms at VGG-I's conv1_1, batch 64; PX = 4 needs 188 registers (one
// block per SM) and took 0.49 ms.
template <int CIN, int PX>
__global__ void __launch_bounds__(256) conv_smallc_fwd_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                                              const float* __restrict__ b, float* __restrict__ y, int N,
                                                              int H, int W, int Cout, int pad, int relu) {
    extern __shared__ float4 smallc_smem[];
    float* ws = reinterpret_cast<float*>(smallc_smem);   // [9*CIN][Cout], then bias [Cout]
    constexpr int K = 9 * CIN;
    // consecutive threads fill consecutive shared words (w is [co][tap][ci])
    for (int i = threadIdx.x; i < K * Cout; i += blockDim.x) ws[i] = w[(i % Cout) * K + i / Cout];
    float* bs = ws + K * Cout;
    for (int i = threadIdx.x; i < Cout; i += blockDim.x) bs[i] = b ? b[i] : 0.f;
    __syncthreads();
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    const int Wp = (Wo + PX - 1) / PX;               // pixel groups per output row
    const int groups = Cout / 16;
    const int P2 = N * Ho * Wp;                      // < 2^31 (checked by the caller)
    const int grp_blocks = (P2 + 31) / 32;           // 32-group warp tasks per channel group
    const int tasks = grp_blocks * groups;
    const int warp_gid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int task = warp_gid; task < tasks; task += warps) {
        const int g = task % groups;
        const int pp = (task / groups) * 32 + lane;
        if (pp >= P2) continue;
        const int ow = (pp % Wp) * PX;
        const int t = pp / Wp;
        const int oh = t % Ho;
        const long long n = t / Ho;
        float in[3][PX + 2][CIN];   // input rows oh-pad .. +2, columns ow-pad .. ow-pad+PX+1
#pragma unroll
        for (int kh = 0; kh < 3; ++kh)
#pragma unroll
            for (int c = 0; c < PX + 2; ++c) {
                const int ih = oh + kh - pad, iw = ow + c - pad;
                const bool ok = ih >= 0 && ih < H && iw >= 0 && iw < W;
#pragma unroll
                for (int ci = 0; ci < CIN; ++ci) in[kh][c][ci] = ok ? __ldg(x + ((n * H + ih) * W + iw) * CIN + ci) : 0.f;
            }
        const int co0 = g * 16;
        float acc[PX][16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float bq = bs[co0 + q];
#pragma unroll
            for (int u = 0; u < PX; ++u) acc[u][q] = bq;
        }
#pragma unroll
        for (int kh = 0; kh < 3; ++kh)
#pragma unroll
            for (int kw = 0; kw < 3; ++kw)
#pragma unroll
                for (int ci = 0; ci < CIN; ++ci) {
                    const float4* wr = reinterpret_cast<const float4*>(ws + ((kh * 3 + kw) * CIN + ci) * Cout + co0);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        const float4 wv = wr[v4];
#pragma unroll
                        for (int u = 0; u < PX; ++u) {
                            const float a = in[kh][kw + u][ci];
                            acc[u][4 * v4 + 0] = fmaf(a, wv.x, acc[u][4 * v4 + 0]);
                            acc[u][4 * v4 + 1] = fmaf(a, wv.y, acc[u][4 * v4 + 1]);
                            acc[u][4 * v4 + 2] = fmaf(a, wv.z, acc[u][4 * v4 + 2]);
                            acc[u][4 * v4 + 3] = fmaf(a, wv.w, acc[u][4 * v4 + 3]);
                        }
                    }
                }
        const long long pix = (n * Ho + oh) * Wo + ow;
#pragma unroll
        for (int u = 0; u < PX; ++u) {
            if (ow + u >= Wo) break;
            float4* dst = reinterpret_cast<float4*>(y + (pix + u) * Cout + co0);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
                float4 o = make_float4(acc[u][4 * v4], acc[u][4 * v4 + 1], acc[u][4 * v4 + 2], acc[u][4 * v4 + 3]);
                if (relu) {
                    o.x = fmaxf(o.x, 0.f);
                    o.y = fmaxf(o.y, 0.f);
                    o.z = fmaxf(o.z, 0.f);
                    o.w = fmaxf(o.w, 0.f);
                }
                __stcs(dst + v4, o);
            }
        }
    }
}

// pixels per thread of the RGB-layer forward
constexpr int kSmallcFwdPx = 2;

int launch_conv_smallc(const float* x, const float* w, const float* b, float* y, int N, int H, int W, int Cin,
                       int Cout, int pad, int relu, cudaStream_t s) {
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    const long long P = static_cast<long long>(N) * Ho * Wo;
    SPRINT_REQUIRE(P < (1ll << 31) - 32, SPRINT_ERR_SHAPE, "conv_fwd: %lld output pixels", P);
    constexpr int PX = kSmallcFwdPx;
    const long long pairs = static_cast<long long>(N) * Ho * ((Wo + PX - 1) / PX);
    const long long total = ((pairs + 31) / 32) * 32 * (Cout / 16);   // threads: one per pixel group and channel group
    const size_t smem = (static_cast<size_t>(9) * Cin * Cout + Cout) * sizeof(float);
    long long g = (total + 255) / 256;
    if (g > 16ll * num_sms()) g = 16ll * num_sms();
    const int grid = static_cast<int>(g < 1 ? 1 : g);
    switch (Cin) {
        case 1: conv_smallc_fwd_kernel<1, PX><<<grid, 256, smem, s>>>(x, w, b, y, N, H, W, Cout, pad, relu); break;
        case 2: conv_smallc_fwd_kernel<2, PX><<<grid, 256, smem, s>>>(x, w, b, y, N, H, W, Cout, pad, relu); break;
        case 3: conv_smallc_fwd_kernel<3, PX><<<grid, 256, smem, s>>>(x, w, b, y, N, H, W, Cout, pad, relu); break;
        default: conv_smallc_fwd_kernel<4, PX><<<grid, 256, smem, s>>>(x, w, b, y, N, H, W, Cout, pad, relu); break;
    }
    return check_launch("conv_smallc_fwd_kernel");
}

// dedw and dedb of a layer with few input channels (the RGB layer) on the CUDA
// cores. As a GEMM it is [Cout] x [9 * Cin] over a k of every output pixel: a
// 27-wide product that would fill few tensor-core columns and need both
// operands re-laid out first. Here one warp takes a segment of kSmallcDwSeg
// output pixels of a row at a time; lane l owns channels l * CPL ..
// l * CPL + CPL - 1. The warp stages the segment's inputs (3 rows of
// kSmallcDwSeg + 2 patch columns, channels padded to 4) and dy rows in its own
// shared buffers with cp.async, one segment ahead of the one it computes (a
// warp's segments are consecutive, so their coordinates advance without a
// division). The 3 x 3 x CIN patch then slides one column per pixel: 3 shared
// loads of a column (one address for the warp) and one of dy per pixel for
// CPL * (9 * CIN + 1) products (the +1: dedb). A block adds its warps' sums in
// warp order in shared memory and writes one partial of Cout * (9 * CIN + 1)
// floats ([co][tap][ci], then [co]); smallc_dw_finish adds the partials in
// block order, so the result depends only on the grid.
constexpr int kSmallcDwSeg = 16;
constexpr int kSmallcDwWarps = 8;
constexpr int kSmallcDwCols = kSmallcDwSeg + 2;      // patch columns of one segment
constexpr int kSmallcDwXs = 3 * kSmallcDwCols * 4;   // staged inputs: [kh][column][4]

// floats of one stage buffer of one warp (inputs, then kSmallcDwSeg dy rows of up to 32 * CPL channels)
constexpr int smallc_dw_stage_floats(int cpl) { return kSmallcDwXs + kSmallcDwSeg * 32 * cpl; }
constexpr size_t smallc_dw_smem(int cpl) {
    return sizeof(float) * 2 * kSmallcDwWarps * static_cast<size_t>(smallc_dw_stage_floats(cpl));
}

// resident blocks per SM (the widest variant holds 2 x 36 + 36 live values per thread)
constexpr int smallc_dw_per_sm(int cin, int cpl) { return cin * cpl > 6 ? 1 : 2; }

int smallc_dw_blocks(int N, int Ho, int Wo, int Cin, int Cout) {
    const long long tasks = static_cast<long long>(N) * Ho * ((Wo + kSmallcDwSeg - 1) / kSmallcDwSeg);
    long long g = (tasks + kSmallcDwWarps - 1) / kSmallcDwWarps;
    const long long cap = static_cast<long long>(smallc_dw_per_sm(Cin, Cout > 32 ? 2 : 1)) * num_sms();
    if (g > cap) g = cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int NPENDING>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(NPENDING) : "memory");
}

// One warp stages the segment at output row r = n * Ho + oh, columns ow0 ..
// ow0 + kSmallcDwSeg - 1, into xs / ds: xs[(kh * cols + c) * 4 + ci] =
// x[n][oh + kh - pad][ow0 - pad + c][ci] (0 outside the image), ds[q * Cout + co]
// = dy[n][oh][ow0 + q][co] (0 past the row's end). A lane copies whole patch
// cells (CIN contiguous floats).
template <int CIN>
__device__ __forceinline__ void smallc_dw_stage(float* xs, float* ds, const float* __restrict__ x,
                                                const float* __restrict__ dy, int n, int oh, int r, int ow0, int H,
                                                int W, int Wo, int Cout, int pad, int lane) {
    for (int cell = lane; cell < 3 * kSmallcDwCols; cell += 32) {
        const int kh = cell / kSmallcDwCols, c = cell - kh * kSmallcDwCols;
        const int ih = oh + kh - pad, iw = ow0 - pad + c;
        float* d = xs + cell * 4;
        if (ih >= 0 && ih < H && iw >= 0 && iw < W) {
            const float* src = x + ((static_cast<long long>(n) * H + ih) * W + iw) * CIN;
#pragma unroll
            for (int ci = 0; ci < CIN; ++ci) cp_async4(d + ci, src + ci);
        } else {
#pragma unroll
            for (int ci = 0; ci < CIN; ++ci) d[ci] = 0.f;
        }
    }
    const int nq = Wo - ow0 < kSmallcDwSeg ? Wo - ow0 : kSmallcDwSeg;
    const float* src = dy + (static_cast<long long>(r) * Wo + ow0) * Cout;
    const int cnt = nq * Cout;
    if ((Cout & 3) == 0) {
        for (int e = lane * 4; e < cnt; e += 128) cp_async16(ds + e, src + e);
    } else {
        for (int e = lane; e < cnt; e += 32) cp_async4(ds + e, src + e);
    }
    for (int e = cnt + lane; e < kSmallcDwSeg * Cout; e += 32) ds[e] = 0.f;
}

template <int CIN, int CPL>
__global__ void __launch_bounds__(kSmallcDwWarps * 32, smallc_dw_per_sm(CIN, CPL))
    conv_smallc_dw_kernel(const float* __restrict__ x, const float* __restrict__ dy, float* __restrict__ partial,
                          int N, int H, int W, int Cout, int pad) {
    constexpr int K = 9 * CIN;
    constexpr int SF = smallc_dw_stage_floats(CPL);
    extern __shared__ float4 smallc_dw_smem_raw[];
    __shared__ float red[32 * CPL * (K + 1)];
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    const int segs = (Wo + kSmallcDwSeg - 1) / kSmallcDwSeg;
    const int tasks = N * Ho * segs;   // < 2^31: the launcher checks the pixel count
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int co0 = lane * CPL;
    const bool live = co0 < Cout;
    float* const stage0 = reinterpret_cast<float*>(smallc_dw_smem_raw) + warp * 2 * SF;
    float acc[CPL][K], accb[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        accb[j] = 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) acc[j][k] = 0.f;
    }
    // warp gw takes the consecutive segments [t0, t1): row-major over (n, oh, segment)
    const long long gw = static_cast<long long>(blockIdx.x) * kSmallcDwWarps + warp;
    const long long nw = static_cast<long long>(gridDim.x) * kSmallcDwWarps;
    const int t0 = static_cast<int>(gw * tasks / nw), t1 = static_cast<int>((gw + 1) * tasks / nw);
    int seg = t0 % segs, r = t0 / segs;   // the next segment to stage; r = n * Ho + oh
    int oh = r % Ho, n = r / Ho;
    auto stage_next = [&](float* buf) {
        smallc_dw_stage<CIN>(buf, buf + kSmallcDwXs, x, dy, n, oh, r, seg * kSmallcDwSeg, H, W, Wo, Cout, pad, lane);
        if (++seg == segs) {
            seg = 0;
            ++r;
            if (++oh == Ho) {
                oh = 0;
                ++n;
            }
        }
    };
    if (t0 < t1) stage_next(stage0);
    cp_async_commit();
    for (int t = t0, b = 0; t < t1; ++t, b ^= 1) {
        if (t + 1 < t1) stage_next(stage0 + (b ^ 1) * SF);
        cp_async_commit();
        cp_async_wait<1>();   // this segment's copies are done; the next one's may still fly
        __syncwarp();
        const float* xs = stage0 + b * SF;
        const float* ds = xs + kSmallcDwXs;
        float win[3][3 * CIN];   // patch columns kw = 0, 1, 2 of the current pixel, [kh][ci]
        auto load_col = [&](float* c, int col) {
#pragma unroll
            for (int kh = 0; kh < 3; ++kh) {
                const float4 v = *reinterpret_cast<const float4*>(xs + (kh * kSmallcDwCols + col) * 4);
                c[kh * CIN + 0] = v.x;
                if constexpr (CIN > 1) c[kh * CIN + 1] = v.y;
                if constexpr (CIN > 2) c[kh * CIN + 2] = v.z;
                if constexpr (CIN > 3) c[kh * CIN + 3] = v.w;
            }
        };
        load_col(win[0], 0);
        load_col(win[1], 1);
#pragma unroll
        for (int q = 0; q < kSmallcDwSeg; ++q) {
            load_col(win[2], q + 2);
            float g[CPL];
#pragma unroll
            for (int j = 0; j < CPL; ++j) g[j] = 0.f;
            if (live) {
                if constexpr (CPL == 2) {
                    const float2 v = *reinterpret_cast<const float2*>(ds + q * Cout + co0);
                    g[0] = v.x;
                    g[1] = v.y;
                } else {
                    g[0] = ds[q * Cout + co0];
                }
            }
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                accb[j] += g[j];
#pragma unroll
                for (int kh = 0; kh < 3; ++kh)
#pragma unroll
                    for (int kw = 0; kw < 3; ++kw)
#pragma unroll
                        for (int ci = 0; ci < CIN; ++ci)
                            acc[j][(kh * 3 + kw) * CIN + ci] =
                                fmaf(g[j], win[kw][kh * CIN + ci], acc[j][(kh * 3 + kw) * CIN + ci]);
            }
#pragma unroll
            for (int c = 0; c < 3 * CIN; ++c) {
                win[0][c] = win[1][c];
                win[1][c] = win[2][c];
            }
        }
        __syncwarp();   // every lane is done with this buffer before it is staged again
    }
    cp_async_wait<0>();
    // the block's sum, warp by warp in warp order: red[co][0..K-1] products, red[co][K] dedb
    for (int w = 0; w < kSmallcDwWarps; ++w) {
        if (warp == w && live) {
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                float* rr = red + (co0 + j) * (K + 1);
#pragma unroll
                for (int k = 0; k < K; ++k) rr[k] = w == 0 ? acc[j][k] : rr[k] + acc[j][k];
                rr[K] = w == 0 ? accb[j] : rr[K] + accb[j];
            }
        }
        __syncthreads();
    }
    const int O = Cout * (K + 1);
    float* part = partial + static_cast<long long>(blockIdx.x) * O;
    for (int i = threadIdx.x; i < O; i += blockDim.x) {
        const bool is_b = i >= Cout * K;
        const int co = is_b ? i - Cout * K : i / K, k = is_b ? K : i % K;
        part[i] = red[co * (K + 1) + k];
    }
}

// dw[o] / db[o - Cout * K] = (accumulate ? old : 0) + alpha * (sum of the
// blocks' partials of output o): 32 outputs per block, 8 block stripes, then
// a fixed pairwise sum of the stripes
__global__ void __launch_bounds__(256) smallc_dw_finish(const float* __restrict__ partial, int nblocks, int Cout, int K,
                                                        float* __restrict__ dw, float* __restrict__ db, float alpha,
                                                        int accumulate) {
    __shared__ float red[8][33];
    const int O = Cout * (K + 1);
    const int lane = threadIdx.x & 31, st = threadIdx.x >> 5;
    const int o = blockIdx.x * 32 + lane;
    const float t = o < O && st < nblocks
                        ? ordered_strided_sum(partial + static_cast<long long>(st) * O + o, (nblocks - st + 7) / 8, 8ll * O)
                        : 0.f;
    red[st][lane] = t;
    __syncthreads();
    if (st != 0 || o >= O) return;
    const float s = ((red[0][lane] + red[1][lane]) + (red[2][lane] + red[3][lane])) +
                    ((red[4][lane] + red[5][lane]) + (red[6][lane] + red[7][lane]));
    if (o < Cout * K) {
        dw[o] = (accumulate ? dw[o] : 0.f) + alpha * s;
    } else if (db) {
        const int c = o - Cout * K;
        db[c] = (accumulate ? db[c] : 0.f) + alpha * s;
    }
}

template <int CIN, int CPL>
int launch_smallc_dw_variant(int grid, const float* x, const float* dy, float* partial, int N, int H, int W, int Cout,
                             int pad, cudaStream_t s) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = smallc_dw_smem(CPL);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(conv_smallc_dw_kernel<CIN, CPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return check_cuda("cudaFuncSetAttribute(conv_smallc_dw_kernel)");
        attr_done[dev] = true;
    }
    conv_smallc_dw_kernel<CIN, CPL><<<grid, kSmallcDwWarps * 32, smem, s>>>(x, dy, partial, N, H, W, Cout, pad);
    return check_launch("conv_smallc_dw_kernel");
}

// Cin <= 4 and Cout <= 64 (Cout even above 32); partial: smallc_dw_blocks() *
// Cout * (9 * Cin + 1) floats
int launch_conv_smallc_dw(const float* x, const float* dy, float* partial, float* dw, float* db, float alpha,
                          int accumulate, int N, int H, int W, int Cin, int Cout, int pad, cudaStream_t s) {
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    const long long P = static_cast<long long>(N) * Ho * Wo;
    SPRINT_REQUIRE(P < (1ll << 31) - 32, SPRINT_ERR_SHAPE, "conv_dW: %lld output pixels", P);
    const int grid = smallc_dw_blocks(N, Ho, Wo, Cin, Cout);
    const bool pairs = Cout > 32;
    int rc;
    switch (Cin) {
        case 1: rc = pairs ? launch_smallc_dw_variant<1, 2>(grid, x, dy, partial, N, H, W, Cout, pad, s)
                           : launch_smallc_dw_variant<1, 1>(grid, x, dy, partial, N, H, W, Cout, pad, s); break;
        case 2: rc = pairs ? launch_smallc_dw_variant<2, 2>(grid, x, dy, partial, N, H, W, Cout, pad, s)
                           : launch_smallc_dw_variant<2, 1>(grid, x, dy, partial, N, H, W, Cout, pad, s); break;
        case 3: rc = pairs ? launch_smallc_dw_variant<3, 2>(grid, x, dy, partial, N, H, W, Cout, pad, s)
                           : launch_smallc_dw_variant<3, 1>(grid, x, dy, partial, N, H, W, Cout, pad, s); break;
        default: rc = pairs ? launch_smallc_dw_variant<4, 2>(grid, x, dy, partial, N, H, W, Cout, pad, s)
                            : launch_smallc_dw_variant<4, 1>(grid, x, dy, partial, N, H, W, Cout, pad, s); break;
    }
    if (rc) return rc;
    const int K = 9 * Cin;
    smallc_dw_finish<<<(Cout * (K + 1) + 31) / 32, 256, 0, s>>>(partial, grid, Cout, K, dw, db, alpha, accumulate);
    return check_launch("smallc_dw_finish");
}

// direct convolution, one thread per output element (co fastest)
__global__ void __launch_bounds__(256) simt_conv_fwd_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                                            const float* __restrict__ b, float* __restrict__ y, int N,
                                                            int H, int W, int Cin, int Cout, int pad, int relu) {
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    const long long total = static_cast<long long>(N) * Ho * Wo * Cout;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int co = static_cast<int>(idx % Cout);
        const long long pix = idx / Cout;
        const int ow = static_cast<int>(pix % Wo);
        const int oh = static_cast<int>((pix / Wo) % Ho);
        const long long n = pix / (static_cast<long long>(Wo) * Ho);
        float acc = b ? b[co] : 0.f;
        for (int kh = 0; kh < 3; ++kh) {
            const int ih = oh + kh - pad;
            if (ih < 0 || ih >= H) continue;
            for (int kw = 0; kw < 3; ++kw) {
                const int iw = ow + kw - pad;
                if (iw < 0 || iw >= W) continue;
                const float* xp = x + ((n * H + ih) * W + iw) * Cin;
                const float* wp = w + (static_cast<long long>(co) * 9 + kh * 3 + kw) * Cin;
                for (int ci = 0; ci < Cin; ++ci) acc = fmaf(xp[ci], wp[ci], acc);
            }
        }
        y[idx] = relu ? fmaxf(acc, 0.f) : acc;
    }
}

__global__ void __launch_bounds__(256) simt_conv_dx_kernel(const float* __restrict__ dy, const float* __restrict__ w,
                                                           const float* __restrict__ relu_src, float* __restrict__ dx,
                                                           int N, int H, int W, int Cin, int Cout, int pad) {
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    const long long total = static_cast<long long>(N) * H * W * Cin;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        if (relu_src && !(relu_src[idx] > 0.f)) {
            dx[idx] = 0.f;
            continue;
        }
        const int ci = static_cast<int>(idx % Cin);
        const long long pix = idx / Cin;
        const int j = static_cast<int>(pix % W);
        const int i = static_cast<int>((pix / W) % H);
        const long long n = pix / (static_cast<long long>(W) * H);
        float acc = 0.f;
        for (int kh = 0; kh < 3; ++kh) {
            const int oh = i - kh + pad;
            if (oh < 0 || oh >= Ho) continue;
            for (int kw = 0; kw < 3; ++kw) {
                const int ow = j - kw + pad;
                if (ow < 0 || ow >= Wo) continue;
                const float* dyp = dy + ((n * Ho + oh) * Wo + ow) * Cout;
                const float* wp = w + (kh * 3 + kw) * static_cast<long long>(Cin) + ci;
                for (int co = 0; co < Cout; ++co) acc = fmaf(dyp[co], wp[static_cast<long long>(co) * 9 * Cin], acc);
            }
        }
        dx[idx] = acc;
    }
}

// partial[chunk][(co*9 + tap)*Cin + ci] = sum over the chunk's output pixels
constexpr int kDwChunk = 512;
__global__ void __launch_bounds__(256) simt_conv_dw_kernel(const float* __restrict__ x, const float* __restrict__ dy,
                                                           float* __restrict__ partial, int N, int H, int W, int Cin,
                                                           int Cout, int pad) {
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    const long long P = static_cast<long long>(N) * Ho * Wo;
    const int O = Cout * 9 * Cin;
    const long long p0 = static_cast<long long>(blockIdx.x) * kDwChunk;
    long long p1 = p0 + kDwChunk;
    if (p1 > P) p1 = P;
    for (int o = threadIdx.x; o < O; o += blockDim.x) {
        const int ci = o % Cin;
        const int tap = (o / Cin) % 9;
        const int co = o / (9 * Cin);
        const int kh = tap / 3, kw = tap % 3;
        float acc = 0.f;
        for (long long pix = p0; pix < p1; ++pix) {
            const int ow = static_cast<int>(pix % Wo);
            const int oh = static_cast<int>((pix / Wo) % Ho);
            const long long n = pix / (static_cast<long long>(Wo) * Ho);
            const int ih = oh + kh - pad, iw = ow + kw - pad;
            if (ih < 0 || ih >= H || iw < 0 || iw >= W) continue;
            acc = fmaf(dy[pix * Cout + co], x[((n * H + ih) * W + iw) * Cin + ci], acc);
        }
        partial[static_cast<long long>(blockIdx.x) * O + o] = acc;
    }
}

// dw[co][tap][ci] = (acc ? dw : 0) + alpha * sum_s partial[tap*S + s][co][ci]
__global__ void dw_split_reduce(const float* __restrict__ partial, int splits, int Cout, int Cin,
                                float* __restrict__ dw, float alpha, int accumulate) {
    const long long total = 9ll * Cout * Cin;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int ci = static_cast<int>(idx % Cin);
        const int tap = static_cast<int>((idx / Cin) % 9);
        const int co = static_cast<int>(idx / (9ll * Cin));
        const float t = ordered_strided_sum(partial + (static_cast<long long>(tap) * splits * Cout + co) * Cin + ci,
                                            splits, static_cast<long long>(Cout) * Cin);
        dw[idx] = (accumulate ? dw[idx] : 0.f) + alpha * t;
    }
}

// dw[co][tap][ci] = (acc ? dw : 0) + alpha * sum_s partial[s][co][tap * rows + ci]
// (taps packed along N, rows >= Cin channel rows per tap)
__global__ void dw_packed_reduce(const float* __restrict__ partial, int splits, int Cout, int Cin, int rows,
                                 float* __restrict__ dw, float alpha, int accumulate) {
    const long long total = 9ll * Cout * Cin;
    const long long np = 9ll * rows;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int ci = static_cast<int>(idx % Cin);
        const int tap = static_cast<int>((idx / Cin) % 9);
        const long long co = idx / (9ll * Cin);
        const float t = ordered_strided_sum(partial + co * np + tap * rows + ci, splits, Cout * np);
        dw[idx] = (accumulate ? dw[idx] : 0.f) + alpha * t;
    }
}

// The factored weight gradient's slabs (Cin = Cout = 64): dw[i] = (acc ? dw : 0) + alpha * sum_s
// slab_s[i], the slabs added in split order
__global__ void dw_fact_reduce(const float* __restrict__ partial, int splits, float* __restrict__ dw, float alpha,
                               int accumulate) {
    constexpr long long slab = 9ll * 64 * 64;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < slab;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float t = ordered_strided_sum(partial + idx, splits, slab);
        dw[idx] = (accumulate ? dw[idx] : 0.f) + alpha * t;
    }
}

__global__ void colsum_finish_k(const float* __restrict__ partial, int chunks, int cols, float* __restrict__ out,
                                float alpha, int accumulate) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= cols) return;
    const float t = ordered_strided_sum(partial + c, chunks, cols);
    out[c] = (accumulate ? out[c] : 0.f) + alpha * t;
}

// The factored convolution's B operand: forward (dx = 0) B'[(dw, co)][(dh, ci)], input
// gradient (dx = 1) B''[(dw, ci)][(dh, co)], both = w[co][dh][dw][ci] (row-major, k fastest)
__global__ void fact_weights_kernel(const float* __restrict__ w, float* __restrict__ out, int Cin, int Cout, int dx) {
    const long long total = 9ll * Cin * Cout;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        int co, ci, dh, dw;
        long long r;
        if (!dx) {   // idx = ((dw * Cout + co) * 3 + dh) * Cin + ci
            ci = static_cast<int>(idx % Cin);
            r = idx / Cin;
            dh = static_cast<int>(r % 3);
            r /= 3;
            co = static_cast<int>(r % Cout);
            dw = static_cast<int>(r / Cout);
        } else {     // idx = ((dw * Cin + ci) * 3 + dh) * Cout + co
            co = static_cast<int>(idx % Cout);
            r = idx / Cout;
            dh = static_cast<int>(r % 3);
            r /= 3;
            ci = static_cast<int>(r % Cin);
            dw = static_cast<int>(r / Cin);
        }
        out[idx] = w[((static_cast<long long>(co) * 3 + dh) * 3 + dw) * Cin + ci];
    }
}

int grid_cap(long long work) {
    long long g = (work + 255) / 256;
    const long long cap = static_cast<long long>(num_sms()) * 16;
    if (g > cap) g = cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

// ------------------------------------------------------------------ plans
inline size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }
inline size_t fbytes(long long n) { return align256(static_cast<size_t>(n) * 4); }

// FC: which GEMMs run on the tensor cores, and the workspace they need.
struct FcPlan {
    bool fwd_tc, dx_tc, dw_tc;
    size_t ws_wT, ws_xT, ws_dyT;  // byte sizes of the transposed copies (offsets follow in this order)
    size_t total() const { return ws_wT + ws_xT + ws_dyT; }
};

FcPlan plan_fc(int N, int in, int out, bool have_wT) {
    FcPlan pl{};
    const bool al = (in % 4 == 0) && (out % 4 == 0);
    pl.fwd_tc = al && in >= 8 && out >= 16;
    pl.dx_tc = al && out >= 8 && in >= 16;
    // dW reads the transposed copies (pitch = batch) and writes dw (pitch = in): out may be anything
    pl.dw_tc = (in % 4 == 0) && (N % 4 == 0) && N >= 8 && in >= 16;
    pl.ws_wT = (pl.dx_tc && !have_wT) ? fbytes(static_cast<long long>(in) * out) : 0;
    pl.ws_xT = pl.dw_tc ? fbytes(static_cast<long long>(N) * in) : 0;
    pl.ws_dyT = pl.dw_tc ? fbytes(static_cast<long long>(N) * out) : 0;
    return pl;
}

struct ConvPlan {
    bool tc = false;
    bool im2col = false;    // forward through an explicit padded im2col + 2-D GEMM
    bool smallc = false;    // Cin <= 4: direct CUDA-core kernel (conv_smallc_fwd_kernel / conv_smallc_dw_kernel)
    int kp = 0;             // padded k of that im2col
    size_t ws_col = 0, ws_wpad = 0;
    Tile tile{};
    PixBox box{};
    int splits = 1, kt_per_split = 0, num_kt = 0;
    size_t ws_wT = 0;       // dedx: transposed weights when the caller has none
    size_t ws_xT = 0, ws_dyT = 0;   // dedw: [C][H][W][N] copies
    size_t ws_partial = 0;  // dedw: split-K partial sums (or the padded output of packed taps)
    size_t ws_colsum = 0;   // dedw: partial bias sums
    int wg_tpt = 0, wg_rows = 0;   // dedw with taps packed along N (0: one tap per tile)
    bool wg_blocked = false;       // dedw copies blocked [H][W*N/32][C][32] (N % 32 == 0)
    bool wg_fact = false;          // dedw factored over kernel rows x columns (Cin = Cout = 64)
    bool rgb = false;              // fwd of the RGB layer (3 -> 64 channels): im2col rows built in shared memory
    bool halo = false;             // fwd / dedx on halo-staged tiles of whole output rows (64 or 128 output channels)
    bool hflip = false;            // that with 128 outputs, weights as M and 256 tile positions as N (one CTA)
    bool fact = false;             // fwd / dedx factored over the kernel columns (64 output channels, wide rows)
    size_t ws_wfact = 0;           // its permuted weights
    GemmPlan gp{};                 // fwd / dedx: tile shape and the k-split of the last, partial round
    size_t ws_tail = 0;            // fwd / dedx: slabs of that split (last in the workspace)
    size_t ws_total() const {
        return ws_wT + ws_xT + ws_dyT + ws_partial + ws_colsum + ws_col + ws_wpad + ws_wfact + ws_tail;
    }
};

// floats per split of the factored weight gradient (Cin = Cout = 64): dW [64][9][64]
constexpr long long wg_fact_slab() { return 9ll * 64 * 64; }

ConvPlan plan_conv(int op, int N, int H, int W, int Cin, int Cout, int pad, bool have_wT) {
    ConvPlan pl;
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    const long long P = static_cast<long long>(N) * Ho * Wo;
    if (op == SPRINT_CONV_FWD && Cin == 3 && Cout == 64 && pad == 1) {
        // the RGB layer: each 128-pixel tile's 27 products per output as one 32-deep k-tile on the
        // tensor cores, its im2col rows written into shared memory by the producer warp (bound by
        // writing y; the CUDA-core kernel below is bound by its shared-memory weight reads)
        pl.tc = pl.rgb = true;
        pl.tile.bn = 64;
        pl.num_kt = 1;
        pl.kt_per_split = 1;
        pl.ws_wpad = fbytes(64ll * TC_BK);
        return pl;
    }
    if (op == SPRINT_CONV_FWD && Cin <= 4 && Cout % 16 == 0 && (9 * Cin + 1) * Cout * 4 <= 48 * 1024) {
        // the RGB layer: direct CUDA-core convolution at output-write speed (no workspace)
        pl.smallc = true;
        return pl;
    }
    if (op == SPRINT_CONV_FWD && Cin % 4 != 0 && Cout % 4 == 0 && Cout >= 16 && 9 * Cin <= 64) {
        // few input channels (the RGB layer): explicit im2col, k padded to 32 or 64
        pl.tc = pl.im2col = true;
        pl.kp = (9 * Cin + 31) / 32 * 32;
        pl.ws_col = fbytes(P * pl.kp);
        pl.ws_wpad = fbytes(static_cast<long long>(Cout) * pl.kp);
        return pl;
    }
    if (op == SPRINT_CONV_FWD || op == SPRINT_CONV_DX) {
        pl.tc = (Cin % 4 == 0) && (Cout % 4 == 0) && Cin >= 8 && Cout >= 16;
        if (!pl.tc) return pl;
        // 64 output channels on rows wide enough for 126-pixel tiles: factored over the kernel
        // columns, a 192-wide GEMM instead of a 64-wide one
        const int nout = op == SPRINT_CONV_FWD ? Cout : Cin, kch = op == SPRINT_CONV_FWD ? Cin : Cout;
        const int fw = op == SPRINT_CONV_FWD ? Wo : W;
        if (pad == 1 && nout == 128 && kch % 32 == 0 && fw + 2 <= HALO_F_POS &&
            (op == SPRINT_CONV_FWD || kch >= 256)) {
            // 128 outputs: tiles of 256 positions (bh rows of the whole row width) against the weights
            // as the 128-row operand, used when they fill >= 80% of the positions (for the input
            // gradient only with >= 8 chunks of reduction: with 4, a tile's MMAs are too short to hide
            // its mask reads, and the tap-by-tap tiles measured faster)
            const int fh = op == SPRINT_CONV_FWD ? Ho : H;
            int bh = HALO_F_POS / (fw + 2);
            if (bh > fh) bh = fh;
            const int th = (fh + bh - 1) / bh;
            const double fill = static_cast<double>(fw) * fh / (static_cast<double>(th) * HALO_F_POS);
            if (halo_f_rows_needed(fw, bh) * 128 <= HALO_F_A_BYTES && fill >= 0.8) {
                pl.tc = pl.halo = pl.hflip = true;
                pl.tile.bn = 128;
                pl.tile.pair = false;
                pl.box = PixBox{fw, bh, 1, 1, th, N};
                pl.num_kt = 9 * (kch / 32);
                pl.kt_per_split = pl.num_kt;
                if (op == SPRINT_CONV_DX && !have_wT) pl.ws_wT = fbytes(9ll * Cin * Cout);
                return pl;
            }
        }
        // (the input gradient with 128 outputs stays tap by tap otherwise: measured faster than the
        // pair tiles below, its ReLU-mask reads weigh more in their epilogue)
        if (pad == 1 && (nout == 64 || (nout == 128 && op == SPRINT_CONV_FWD)) && kch % 32 == 0) {
            // halo-staged tiles: bh output rows of bw pixels (bw + 2 <= 115, so a 128-row MMA
            // covers them and the buffer fits its stage), used when they fill >= 80% of the rows
            const int fh = op == SPRINT_CONV_FWD ? Ho : H;
            const int per_row = (fw + 112) / 113;
            const int bw = (fw + per_row - 1) / per_row;
            int bh = per_row == 1 ? TC_BM / (bw + 2) : 1;
            if (bh > fh) bh = fh;
            const int th = (fh + bh - 1) / bh;
            const double fill = static_cast<double>(fw) * fh / (static_cast<double>(per_row) * th * TC_BM);
            if (bh >= 1 && halo_rows_needed(bw, bh) <= HALO_A_ROWS && fill >= 0.8) {
                // 64 outputs: factored over the kernel columns (a 192-wide MMA on permuted weights)
                pl.halo = true;
                pl.tile.bn = nout == 64 ? 192 : 128;
                pl.tile.pair = true;
                pl.box = PixBox{bw, bh, 1, per_row, th, N};
                pl.num_kt = 9 * (kch / 32);
                pl.kt_per_split = pl.num_kt;
                if (nout == 64)
                    pl.ws_wfact = fbytes(9ll * nout * kch);
                else if (op == SPRINT_CONV_DX && !have_wT)
                    pl.ws_wT = fbytes(9ll * Cin * Cout);
                return pl;
            }
        }
        if (pad == 1 && nout == 64 && kch % 32 == 0 && fw >= 96) {
            pl.fact = true;
            pl.tile.bn = 192;
            pl.tile.pair = true;
            pl.num_kt = 3 * (kch / 32);
            pl.kt_per_split = pl.num_kt;
            pl.box = PixBox{TC_FACT_OUT, 1, 1, (fw + TC_FACT_OUT - 1) / TC_FACT_OUT, op == SPRINT_CONV_FWD ? Ho : H, N};
            pl.ws_wfact = fbytes(3ll * nout * 3 * kch);
            return pl;
        }
        const int gw = op == SPRINT_CONV_FWD ? Wo : W, gh = op == SPRINT_CONV_FWD ? Ho : H;
        pl.box = pick_box(TC_BM, gw, gh, N);
        const int ncols = op == SPRINT_CONV_FWD ? Cout : Cin;
        pl.num_kt = 9 * (((op == SPRINT_CONV_FWD ? Cin : Cout) + 31) / 32);
        pl.gp = plan_gemm(pl.box.tiles(), ncols, 1, ncols >= 256 ? 256 : (ncols >= 128 ? 128 : 64), pl.num_kt, true);
        pl.tile = pl.gp.tile;
        pl.ws_tail = pl.gp.tail_splits > 1 ? tail_bytes() : 0;
        pl.kt_per_split = pl.num_kt;
        if (op == SPRINT_CONV_DX && !have_wT) pl.ws_wT = fbytes(9ll * Cin * Cout);
        return pl;
    }
    // dedw
    if (Cin <= 4 && Cout <= 64 && (Cout <= 32 || Cout % 2 == 0)) {
        // the RGB layer: direct CUDA-core kernel, dedb in the same pass
        pl.smallc = true;
        pl.ws_partial = fbytes(static_cast<long long>(smallc_dw_blocks(N, Ho, Wo, Cin, Cout)) * Cout * (9 * Cin + 1));
        return pl;
    }
    // x^T puts channels outermost, so any Cin works; outputs with Cin % 4 != 0
    // are written with direct stores
    pl.tc = (N % 4 == 0) && (Cout % 4 == 0) && Cout >= 16;
    // dedb: partial column sums of the dy transpose (one per pixel and 32-image
    // tile and channel) on the tensor-core path, else chunks of colsum
    const int chunks = colsum_chunks(P, Cout);
    pl.ws_colsum = pl.tc ? fbytes(static_cast<long long>(Cout) * Ho * Wo * ((N + 31) / 32))
                         : (chunks > 1 ? fbytes(static_cast<long long>(chunks) * Cout) : 0);
    if (!pl.tc) {
        const long long nchunk = (P + kDwChunk - 1) / kDwChunk;
        pl.ws_partial = fbytes(nchunk * Cout * 9 * Cin);
        return pl;
    }
    pl.ws_xT = fbytes(static_cast<long long>(N) * H * W * Cin);
    pl.ws_dyT = fbytes(P * Cout);
    pl.wg_blocked = N % 32 == 0;
    pl.box = PixBox{0, 0, 0, static_cast<int>((static_cast<long long>(Wo) * N + TC_BK - 1) / TC_BK), Ho, 1};
    pl.num_kt = pl.box.tw * Ho;   // per output row: ceil(Wo*N / 32) k-tiles
    const long long m_tiles = (Cout + TC_BM - 1) / TC_BM;
    const bool pair_m = m_tiles >= 2 && (m_tiles % 2 == 0 || m_tiles >= 6);
    long long base;
    if (pl.wg_blocked && Cin == 64 && Cout == 64 && pad == 1) {
        // Cout = 64 would fill half of every 128-row tile: D = [(dh, ci)] x [(dw, co)] on a
        // CTA pair (192 of its 256 rows used, all nine taps from 9 boxes per k-tile), one unit
        // per k split
        pl.wg_fact = true;
        pl.tile.bn = 192;
        pl.tile.pair = true;
        base = 1;
    } else if (Cin <= 128 && (Cin % 8 == 0 || Cin < 8)) {
        // Few input channels: an n-tile holds whole taps (rows of x^T at their
        // shifts), wg_rows rows each (8 for Cin < 8: the box rows past Cin are TMA
        // zero fill), instead of one tap of a few columns; D = [Cout][9 * wg_rows].
        pl.wg_rows = Cin < 8 ? 8 : Cin;
        const int rows = pl.wg_rows;
        int bn = 0;
        if (9 * rows <= 256) {   // every tap in one tile: the narrowest width that holds 9 * rows
            const int cands[5] = {64, 128, 160, 192, 256};
            for (int i = 0; i < 5 && !bn; ++i)
                if (cands[i] >= 9 * rows && cands[i] % rows == 0) bn = cands[i];
        }
        bool pair = false;
        if (!bn) {
            // several tiles: least (tiles x width) / efficiency over the widths that hold whole taps
            const int cands[4] = {256, 192, 160, 128};
            const double eff[4] = {0.86, 0.72, 0.68, 0.58}, eff_pair[4] = {1.0, 0.79, 0.86, 0.74};
            double best_c = 1e300;
            for (int i = 0; i < 4; ++i) {
                const int c = cands[i];
                if (c % rows) continue;
                const bool pr = pair_m && (c / 2) % rows == 0;
                const double cost = static_cast<double>((9 + c / rows - 1) / (c / rows)) * c / (pr ? eff_pair[i] : eff[i]);
                if (cost < best_c - 1e-9) {
                    best_c = cost;
                    bn = c;
                    pair = pr;
                }
            }
        } else {
            pair = pair_m && (bn / 2) % rows == 0;
        }
        pl.tile.bn = bn;
        pl.tile.pair = pair;
        pl.wg_tpt = bn / rows;
        base = (pl.tile.pair ? (m_tiles + 1) / 2 : m_tiles) * ((9 + pl.wg_tpt - 1) / pl.wg_tpt);
    } else {
        // split-K below fills the machine, so the widest tile (best MMA shape) is used,
        // on CTA pairs when Cout spans an even number of 128-row tiles (or many)
        pl.tile.bn = Cin > 128 ? 256 : (Cin > 64 ? 128 : 64);
        pl.tile.pair = pair_m;
        base = (pl.tile.pair ? (m_tiles + 1) / 2 : m_tiles) * ((Cin + pl.tile.bn - 1) / pl.tile.bn) * 9;
    }
    const long long slots = pl.tile.pair ? num_sms() / 2 : num_sms();
    // split count: fewest (rounds of units) x (k-tiles per unit), counting each
    // split's partial-sum write and read as ~8 k-tiles of work; splits keep >= 8 k-tiles
    long long maxs = pl.num_kt / 8;
    if (maxs < 1) maxs = 1;
    long long want = 1;
    double best = 1e300;
    for (long long sp = 1; sp <= maxs && sp <= 4 * slots; ++sp) {
        const long long per = (pl.num_kt + sp - 1) / sp;
        const long long rounds = (base * sp + slots - 1) / slots;
        const double cost = static_cast<double>(rounds) * (per + (sp > 1 ? 8 : 0));
        if (cost < best - 1e-9) {
            best = cost;
            want = sp;
        }
    }
    pl.kt_per_split = static_cast<int>((pl.num_kt + want - 1) / want);
    pl.splits = (pl.num_kt + pl.kt_per_split - 1) / pl.kt_per_split;
    if (pl.wg_fact) {
        pl.ws_partial = fbytes(static_cast<long long>(pl.splits) * wg_fact_slab());
    } else if (pl.wg_tpt > 0) {
        if (pl.splits > 1 || pl.wg_rows != Cin)
            pl.ws_partial = fbytes(static_cast<long long>(pl.splits) * Cout * 9 * pl.wg_rows);
    } else if (pl.splits > 1) {
        pl.ws_partial = fbytes(static_cast<long long>(pl.splits) * 9 * Cout * Cin);
    }
    return pl;
}

int check_conv_shape(const char* fn, int N, int H, int W, int Cin, int Cout, int pad) {
    SPRINT_REQUIRE(N >= 1 && Cin >= 1 && Cout >= 1 && (pad == 0 || pad == 1) && H + 2 * pad >= 3 && W + 2 * pad >= 3,
                   SPRINT_ERR_SHAPE, "%s: bad shape N=%d H=%d W=%d Cin=%d Cout=%d pad=%d", fn, N, H, W, Cin, Cout,
                   pad);
    SPRINT_REQUIRE(N <= (1 << 24) && H <= 32768 && W <= 32768 && Cin <= (1 << 20) && Cout <= (1 << 20),
                   SPRINT_ERR_SHAPE, "%s: dimension too large", fn);
    SPRINT_REQUIRE(static_cast<long long>(H) * W <= 65535, SPRINT_ERR_SHAPE, "%s: H*W > 65535 not supported", fn);
    return SPRINT_OK;
}

int check_ws(const char* fn, const void* ws, size_t ws_bytes, size_t need) {
    SPRINT_REQUIRE(need == 0 || (ws && ws_bytes >= need), SPRINT_ERR_WORKSPACE,
                   "%s: needs a workspace of %zu bytes (got %zu)", fn, need, ws ? ws_bytes : static_cast<size_t>(0));
    SPRINT_REQUIRE(ws == nullptr || aligned16(ws), SPRINT_ERR_ALIGN, "%s: workspace not 16-byte aligned", fn);
    return SPRINT_OK;
}

// D[M][N] (epilogue) = A[M][K] . B[N][K]^T on the tensor cores; false if the
// tensor maps cannot describe the operands (the caller then uses CUDA cores).
bool gemm2d_tc(const float* A, long long lda, const float* B, long long ldb, int M, int N, int K, TcParams p,
               cudaStream_t s, int* rc) {
    const long long m_tiles = (M + TC_BM - 1) / TC_BM;
    const Tile tl = pick_tile(m_tiles, N, 1, N >= 256 ? 256 : (N >= 128 ? 128 : 64));
    CUtensorMap ta, tb, td;
    const uint64_t da[2] = {(uint64_t)K, (uint64_t)M}, sa[1] = {(uint64_t)lda * 4};
    const uint64_t db[2] = {(uint64_t)K, (uint64_t)N}, sb[1] = {(uint64_t)ldb * 4};
    const uint32_t ba[2] = {32, 128}, bb[2] = {32, tl.b_rows()};
    if (!make_tmap(&ta, A, 2, da, sa, ba) || !make_tmap(&tb, B, 2, db, sb, bb)) return false;
    // TMA store of D when its row pitch is a multiple of 16 bytes, else direct stores
    p.store = ST_DIRECT;
    td = ta;
    if ((p.ldd & 3) == 0 && aligned16(p.D)) {
        const uint64_t dd[2] = {(uint64_t)N, (uint64_t)M}, sd[1] = {(uint64_t)p.ldd * 4};
        const uint32_t bd[2] = {32, 32};
        if (make_tmap(&td, p.D, 2, dd, sd, bd, false)) p.store = ST_2D;
    }
    p.M = M;
    p.N = N;
    p.num_kt = (K + TC_BK - 1) / TC_BK;
    p.kt_per_split = p.num_kt;
    *rc = launch_tc<ROLE_GEMM_2D>(tl, ta, tb, td, p, m_tiles, (N + tl.bn - 1) / tl.bn, 1, s);
    return true;
}

// Grouped form: D_g (epilogue) = A_g . B_g^T for g < G, every problem of the
// same shape, kMaxGroup problems per launch; per-problem bias / mask / D come
// from the arrays (bias and mask may be null arrays). Every tensor map is made
// before the first launch; false if one cannot be (nothing launched then).
bool gemm2d_tc_group(const float* const* A, long long lda, const float* const* B, long long ldb, int M, int N, int K,
                     TcParams p, const float* const* bias, const float* const* mask, float* const* D, int G,
                     cudaStream_t s, int* rc, float* tail_ws = nullptr, size_t tail_ws_bytes = 0,
                     float* const* DT = nullptr, float* const* vec = nullptr) {
    *rc = SPRINT_OK;
    if (G <= 0) return true;
    const long long m_tiles = (M + TC_BM - 1) / TC_BM;
    const int per_launch = G < kMaxGroup ? G : kMaxGroup;
    const int num_kt = (K + TC_BK - 1) / TC_BK;
    const bool tail_ok = tail_ws && tail_ws_bytes >= tail_bytes() && aligned16(tail_ws);
    // the tail split is planned for a full launch of per_launch problems (the last chunk may hold fewer)
    const GemmPlan plan = plan_gemm(m_tiles, N, per_launch, N >= 256 ? 256 : (N >= 128 ? 128 : 64), num_kt, tail_ok);
    const Tile tl = plan.tile;
    const uint64_t da[2] = {(uint64_t)K, (uint64_t)M}, sa[1] = {(uint64_t)lda * 4};
    const uint64_t db[2] = {(uint64_t)K, (uint64_t)N}, sb[1] = {(uint64_t)ldb * 4};
    const uint32_t ba[2] = {32, 128}, bb[2] = {32, tl.b_rows()};
    // D holds the columns before the vector column (p.vec_col, with vec), all N otherwise
    if (!vec) p.vec_col = -1;
    const uint64_t dd[2] = {(uint64_t)(p.vec_col >= 0 ? p.vec_col : N), (uint64_t)M}, sd[1] = {(uint64_t)p.ldd * 4};
    const uint32_t bd[2] = {32, 32};
    bool tma_store = (p.ldd & 3) == 0;
    for (int g = 0; g < G && tma_store; ++g) tma_store = aligned16(D[g]);
    const int chunks = (G + kMaxGroup - 1) / kMaxGroup;
    std::vector<TcMaps<kMaxGroup>> maps(chunks);
    for (int g = 0; g < G; ++g) {
        TcMaps<kMaxGroup>& m = maps[g / kMaxGroup];
        const int i = g % kMaxGroup;
        if (!make_tmap(&m.a[i], A[g], 2, da, sa, ba) || !make_tmap(&m.b[i], B[g], 2, db, sb, bb)) return false;
        if (tma_store) {
            if (!make_tmap(&m.d[i], D[g], 2, dd, sd, bd, false)) return false;
        } else {
            m.d[i] = m.a[i];
        }
    }
    p.store = tma_store ? ST_2D : ST_DIRECT;
    p.M = M;
    p.N = N;
    p.num_kt = (K + TC_BK - 1) / TC_BK;
    p.kt_per_split = p.num_kt;
    // problems that share B (replicas reading one weight version): units of one
    // n-tile of all problems together, so a B tile is read from HBM once and then
    // from L2 (A, re-read per n-tile, is the small operand here)
    p.z_mid = 0;
    for (int g = 1; g < G && !p.z_mid; ++g)
        for (int h = 0; h < g; ++h)
            if (B[g] == B[h]) p.z_mid = 1;
    const long long n_tiles = (N + tl.bn - 1) / tl.bn;
    const long long m_units = tl.pair ? (m_tiles + 1) / 2 : m_tiles;
    for (int c = 0; c < chunks; ++c) {
        const int g0 = c * kMaxGroup, n = G - g0 < kMaxGroup ? G - g0 : kMaxGroup;
        for (int i = 0; i < kMaxGroup; ++i) {
            p.g_bias[i] = (i < n && bias) ? bias[g0 + i] : nullptr;
            p.g_mask[i] = (i < n && mask) ? mask[g0 + i] : nullptr;
            p.g_D[i] = i < n ? D[g0 + i] : nullptr;
            p.g_DT[i] = (i < n && DT) ? DT[g0 + i] : nullptr;
            p.g_vec[i] = (i < n && vec) ? vec[g0 + i] : nullptr;
        }
        const long long units = m_units * n_tiles * n;
        p.tail_splits = 1;
        if (plan.tail_splits > 1 && units > plan.tail_start) {
            p.tail_splits = plan.tail_splits;
            p.tail_kt = plan.tail_kt;
            p.tail_start = static_cast<int>(plan.tail_start);
            p.tail_part = tail_ws;
        }
        *rc = launch_tc_maps<ROLE_GEMM_2D, kMaxGroup>(tl, maps[c], p, m_tiles, n_tiles, n, s);
        if (*rc) return true;
        if (p.tail_splits > 1 && (*rc = launch_tail_reduce<ROLE_GEMM_2D>(plan, p, m_units, n_tiles, n, s)))
            return true;
    }
    return true;
}

// pointer-array arguments of the batched entry points
int check_ptr_array(const char* fn, const char* what, const void* const* arr, int batch, bool array_nullable,
                    bool entries_nullable) {
    if (!arr) {
        SPRINT_REQUIRE(array_nullable, SPRINT_ERR_INVALID_ARG, "%s: %s is NULL", fn, what);
        return SPRINT_OK;
    }
    for (int g = 0; g < batch; ++g) {
        SPRINT_REQUIRE(entries_nullable || arr[g], SPRINT_ERR_INVALID_ARG, "%s: %s[%d] is NULL", fn, what, g);
        SPRINT_REQUIRE(!arr[g] || aligned16(arr[g]), SPRINT_ERR_ALIGN, "%s: %s[%d] not 16-byte aligned", fn, what, g);
    }
    return SPRINT_OK;
}

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

}  // namespace
}  // namespace sprint

using namespace sprint;

// ====================================================================== FC
extern "C" size_t sprint_fc_workspace_size(int N, int in, int out, int have_wT) {
    if (N < 1 || in < 1 || out < 1) return 0;
    return plan_fc(N, in, out, have_wT != 0).total();
}

extern "C" int sprint_fc_fwd(const float* x, const float* w, const float* b, float* y, int N, int in, int out,
                             int relu, sprint_stream_t stream) {
    SPRINT_REQUIRE(N >= 1 && in >= 1 && out >= 1, SPRINT_ERR_SHAPE, "%s: need N, in, out >= 1 (got %d, %d, %d)",
                   __func__, N, in, out);
    SPRINT_NONNULL(x, "x");
    SPRINT_NONNULL(w, "w");
    SPRINT_NONNULL(y, "y");
    SPRINT_ALIGNED(x, "x");
    SPRINT_ALIGNED(w, "w");
    SPRINT_ALIGNED(b, "b");
    SPRINT_ALIGNED(y, "y");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const FcPlan pl = plan_fc(N, in, out, true);
    if (pl.fwd_tc) {
        TcParams p = base_params();
        p.epi = EPI_STORE;
        p.D = y;
        p.ldd = out;
        p.bias = b;
        p.relu = relu;
        int rc = SPRINT_OK;
        if (gemm2d_tc(x, in, w, in, N, out, in, p, s, &rc)) return rc;
    }
    if (out <= kSkinnyN) {
        if (in % 4 == 0) return launch_skinny4(&x, &w, &b, &y, 1, N, out, in, relu, s);
        skinny_nt_kernel<<<(N + 1) / 2, 256, 0, s>>>(x, in, w, in, b, y, out, N, out, in, relu);
        return check_launch("skinny_nt_kernel");
    }
    SimtGemm g{N, out, in, x, in, 1, w, in, 1, y, out, b, nullptr, 0, 1.f, 0, relu, SIMT_STORE};
    return launch_simt_gemm(g, s);
}

extern "C" int sprint_fc_bwd(const float* x, const float* w, const float* wT, const float* dy, const float* relu_src,
                             float* dx, float* dw, float* db, float alpha, int accumulate, int N, int in, int out,
                             void* ws, size_t ws_bytes, sprint_stream_t stream) {
    SPRINT_REQUIRE(N >= 1 && in >= 1 && out >= 1, SPRINT_ERR_SHAPE, "%s: need N, in, out >= 1 (got %d, %d, %d)",
                   __func__, N, in, out);
    SPRINT_NONNULL(x, "x");
    SPRINT_NONNULL(w, "w");
    SPRINT_NONNULL(dy, "dy");
    SPRINT_NONNULL(dw, "dw");
    SPRINT_ALIGNED(x, "x");
    SPRINT_ALIGNED(w, "w");
    SPRINT_ALIGNED(wT, "wT");
    SPRINT_ALIGNED(dy, "dy");
    SPRINT_ALIGNED(relu_src, "relu_src");
    SPRINT_ALIGNED(dx, "dx");
    SPRINT_ALIGNED(dw, "dw");
    SPRINT_ALIGNED(db, "db");
    FcPlan pl = plan_fc(N, in, out, wT != nullptr);
    if (!dx) pl.ws_wT = 0;
    int rc = check_ws(__func__, ws, ws_bytes, pl.total());
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* wsb = static_cast<char*>(ws);
    float* ws_wT = reinterpret_cast<float*>(wsb);
    float* xT = reinterpret_cast<float*>(wsb + pl.ws_wT);
    float* dyT = reinterpret_cast<float*>(wsb + pl.ws_wT + pl.ws_xT);

    // dedx fc: dx = mask * (dy . w) = mask * (dy . (w^T)^T)
    if (dx) {
        bool done = false;
        if (pl.dx_tc) {
            const float* wt = wT;
            if (!wt) {
                if ((rc = launch_transpose(w, ws_wT, 1, out, in, 0, in, 0, out, s))) return rc;
                wt = ws_wT;
            }
            TcParams p = base_params();
            p.epi = EPI_MASK;
            p.D = dx;
            p.ldd = in;
            p.mask = relu_src;
            p.ldm = in;
            done = gemm2d_tc(dy, out, wt, out, N, in, out, p, s, &rc);
            if (rc) return rc;
        }
        if (!done && out <= 32) {
            if (in % 4 == 0) {
                if ((rc = launch_smallk_dx4(&dy, &w, relu_src ? &relu_src : nullptr, &dx, nullptr, 1, N, in, out, s)))
                    return rc;
            } else {
                smallk_dx_kernel<<<grid_cap(static_cast<long long>(N) * in), 256, 0, s>>>(dy, w, relu_src, dx, N,
                                                                                         in, out);
                if ((rc = check_launch("smallk_dx_kernel"))) return rc;
            }
            done = true;
        }
        if (!done) {
            SimtGemm g{N, in, out, dy, out, 1, w, 1, in, dx, in, nullptr, relu_src, in, 1.f, 0, 0, SIMT_MASK};
            if ((rc = launch_simt_gemm(g, s))) return rc;
        }
    }
    // dedw: dw = acc*dw + alpha * (dy^T) . (x^T)^T, contracting over the batch
    {
        bool done = false;
        if (pl.dw_tc) {
            if ((rc = launch_transpose(x, xT, 1, N, in, 0, in, 0, N, s))) return rc;
            if ((rc = launch_transpose(dy, dyT, 1, N, out, 0, out, 0, N, s))) return rc;
            TcParams p = base_params();
            p.epi = EPI_ACCUM;
            p.D = dw;
            p.ldd = in;
            p.alpha = alpha;
            p.accumulate = accumulate;
            done = gemm2d_tc(dyT, N, xT, N, out, in, N, p, s, &rc);
            if (rc) return rc;
        }
        if (!done) {
            SimtGemm g{out, in, N, dy, 1, out, x, 1, in, dw, in, nullptr, nullptr, 0, alpha, accumulate, 0, SIMT_ACCUM};
            if ((rc = launch_simt_gemm(g, s))) return rc;
        }
    }
    // dedb
    if (db && (rc = launch_colsum(dy, N, out, nullptr, db, alpha, accumulate, s))) return rc;
    return SPRINT_OK;
}

// ====================================================================== FC, batched over problems
extern "C" size_t sprint_fc_batched_workspace_size(int batch, int N, int in, int out, int have_wT) {
    if (batch < 1 || N < 1 || in < 1 || out < 1) return 0;
    return static_cast<size_t>(batch) * round256(plan_fc(N, in, out, have_wT != 0).total()) + tail_bytes();
}

extern "C" size_t sprint_fc_fwd_batched_workspace_size(void) { return tail_bytes(); }

extern "C" int sprint_fc_fwd_batched(const float* const* x, const float* const* w, const float* const* b,
                                     float* const* y, float* const* yT, int batch, int N, int in, int out, int relu,
                                     void* ws, size_t ws_bytes, sprint_stream_t stream) {
    SPRINT_REQUIRE(batch >= 0 && N >= 1 && in >= 1 && out >= 1, SPRINT_ERR_SHAPE,
                   "%s: need batch >= 0 and N, in, out >= 1 (got %d, %d, %d, %d)", __func__, batch, N, in, out);
    if (batch == 0) return SPRINT_OK;
    int rc;
    if ((rc = check_ptr_array(__func__, "x", reinterpret_cast<const void* const*>(x), batch, false, false)) ||
        (rc = check_ptr_array(__func__, "w", reinterpret_cast<const void* const*>(w), batch, false, false)) ||
        (rc = check_ptr_array(__func__, "b", reinterpret_cast<const void* const*>(b), batch, true, true)) ||
        (rc = check_ptr_array(__func__, "y", reinterpret_cast<const void* const*>(y), batch, false, false)) ||
        (rc = check_ptr_array(__func__, "yT", reinterpret_cast<const void* const*>(yT), batch, true, false)))
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // grouped tensor-core launch; narrow outputs (e.g. a 10-way classifier, out % 4 != 0) too
    // when the last-round k split is available (few tiles, long k): direct stores write y
    // (and the transposed copy, rows of N, when asked for)
    const bool tail_room = ws && ws_bytes >= tail_bytes();
    bool done = false;
    if (batch > 1 && (plan_fc(N, in, out, true).fwd_tc || (in % 4 == 0 && in >= 256 && tail_room))) {
        TcParams p = base_params();
        p.epi = EPI_STORE;
        p.ldd = out;
        p.relu = relu;
        p.lddT = N;
        done = gemm2d_tc_group(x, in, w, in, N, out, in, p, b, nullptr, y, batch, s, &rc, static_cast<float*>(ws),
                               ws_bytes, yT);
        if (rc) return rc;
        if (done) return SPRINT_OK;
    }
    if (out <= kSkinnyN && in % 4 == 0) {
        if ((rc = launch_skinny4(x, w, b, y, batch, N, out, in, relu, s))) return rc;
    } else {
        for (int g = 0; g < batch; ++g)
            if ((rc = sprint_fc_fwd(x[g], w[g], b ? b[g] : nullptr, y[g], N, in, out, relu, stream))) return rc;
    }
    // paths without the transposed store: transpose the result
    if (yT) return launch_transpose_group(const_cast<const float* const*>(y), yT, batch, N, out, s);
    return SPRINT_OK;
}

// the parameter-server update of one FC layer over the batch's GradBufs
struct PsArgs {
    int opt;
    const float* w_in;
    const float* b_in;
    float* w_out;
    float* b_out;
    float* wT_out;
    float* w_state;
    float* b_state;
    float eta, hp, wd;
};

static int fc_bwd_batched_impl(const char* fn, const float* const* x, const float* const* xT1, const float* const* w,
                               const float* const* wT, const float* const* dy, const float* const* dyT,
                               const float* const* relu_src, float* const* dx, float* const* dxT, float* const* dw,
                               float* const* db, float alpha, int accumulate, int batch, int N, int in, int out,
                               void* ws, size_t ws_bytes, sprint_stream_t stream, const PsArgs* ps) {
    SPRINT_REQUIRE(batch >= 0 && N >= 1 && in >= 1 && out >= 1, SPRINT_ERR_SHAPE,
                   "%s: need batch >= 0 and N, in, out >= 1 (got %d, %d, %d, %d)", fn, batch, N, in, out);
    if (batch == 0) return SPRINT_OK;
    int rc;
    if ((rc = check_ptr_array(fn, "x", reinterpret_cast<const void* const*>(x), batch, false, false)) ||
        (rc = check_ptr_array(fn, "xT1", reinterpret_cast<const void* const*>(xT1), batch, true, false)) ||
        (rc = check_ptr_array(fn, "w", reinterpret_cast<const void* const*>(w), batch, false, false)) ||
        (rc = check_ptr_array(fn, "wT", reinterpret_cast<const void* const*>(wT), batch, true, false)) ||
        (rc = check_ptr_array(fn, "dy", reinterpret_cast<const void* const*>(dy), batch, false, false)) ||
        (rc = check_ptr_array(fn, "dyT", reinterpret_cast<const void* const*>(dyT), batch, true, false)) ||
        (rc = check_ptr_array(fn, "relu_src", reinterpret_cast<const void* const*>(relu_src), batch, true,
                              true)) ||
        (rc = check_ptr_array(fn, "dx", reinterpret_cast<const void* const*>(dx), batch, true, false)) ||
        (rc = check_ptr_array(fn, "dxT", reinterpret_cast<const void* const*>(dxT), batch, true, false)) ||
        (rc = check_ptr_array(fn, "dw", reinterpret_cast<const void* const*>(dw), batch, false, false)) ||
        (rc = check_ptr_array(fn, "db", reinterpret_cast<const void* const*>(db), batch, true, false)))
        return rc;
    SPRINT_REQUIRE(!dxT || dx, SPRINT_ERR_INVALID_ARG, "%s: dxT needs dx", fn);
    FcPlan pl = plan_fc(N, in, out, wT != nullptr);
    if (!dx) pl.ws_wT = 0;
    const size_t per = round256(pl.total());
    if ((rc = check_ws(fn, ws, ws_bytes, per * batch))) return rc;
    // what follows the per-problem slices serves the tail split of the GEMMs (optional)
    float* tail_ws = ws ? reinterpret_cast<float*>(static_cast<char*>(ws) + per * batch) : nullptr;
    const size_t tail_ws_bytes = ws ? ws_bytes - per * batch : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (ps) {
        SPRINT_REQUIRE(ps->opt >= PS_SGD && ps->opt <= PS_NESTEROV, SPRINT_ERR_INVALID_ARG,
                       "%s: unknown update rule %d", fn, ps->opt);
        SPRINT_REQUIRE(batch <= kMaxGroup, SPRINT_ERR_UNSUPPORTED, "%s: the update sums at most %d GradBufs (got %d)",
                       fn, kMaxGroup, batch);
        SPRINT_REQUIRE(ps->w_in && ps->w_out && (ps->opt == PS_SGD || ps->w_state), SPRINT_ERR_INVALID_ARG,
                       "%s: NULL w_in, w_out or w_state", fn);
        SPRINT_REQUIRE(!db || (ps->b_in && ps->b_out && (ps->opt == PS_SGD || ps->b_state)), SPRINT_ERR_INVALID_ARG,
                       "%s: NULL b_in, b_out or b_state", fn);
        SPRINT_REQUIRE(aligned16(ps->w_in) && aligned16(ps->w_out) && (!ps->w_state || aligned16(ps->w_state)) &&
                           (!ps->wT_out || aligned16(ps->wT_out)) && (!ps->b_in || aligned16(ps->b_in)) &&
                           (!ps->b_out || aligned16(ps->b_out)) && (!ps->b_state || aligned16(ps->b_state)),
                       SPRINT_ERR_ALIGN, "%s: update pointers must be 16-byte aligned", fn);
    }
    // the update by the standalone kernels (what the weight-gradient GEMM did not fuse)
    // the layer's update after its backward pass (in stream order): W' (and W'^T in
    // the same pass), then b'
    auto finish_ps = [&]() -> int {
        if (!ps) return SPRINT_OK;
        int r;
        const float* const* bufs = const_cast<const float* const*>(dw);
        if (ps->wT_out)
            r = launch_ps_update_t(ps->opt, fn, ps->w_in, ps->w_out, ps->wT_out, ps->w_state, bufs, batch, out, in,
                                   static_cast<size_t>(out) * in, ps->eta, ps->hp, ps->wd, stream);
        else
            r = launch_ps_update(ps->opt, fn, ps->w_in, ps->w_out, ps->w_state, bufs, batch,
                                 static_cast<size_t>(out) * in, ps->eta, ps->hp, ps->wd, stream);
        if (r) return r;
        if (db)
            return launch_ps_update(ps->opt, fn, ps->b_in, ps->b_out, ps->b_state, const_cast<const float* const*>(db),
                                    batch, static_cast<size_t>(out), ps->eta, ps->hp, ps->wd, stream);
        return SPRINT_OK;
    };
    const bool extras = xT1 || dyT || dxT;
    if (batch == 1 && !extras) {
        if ((rc = sprint_fc_bwd(x[0], w[0], wT ? wT[0] : nullptr, dy[0], relu_src ? relu_src[0] : nullptr,
                                dx ? dx[0] : nullptr, dw[0], db ? db[0] : nullptr, alpha, accumulate, N, in, out, ws,
                                ws_bytes, stream)))
            return rc;
        return finish_ps();
    }
    char* wsb = static_cast<char*>(ws);
    std::vector<float*> ws_wT(batch), xT(batch), dyT_ws(batch);
    for (int g = 0; g < batch; ++g) {
        ws_wT[g] = reinterpret_cast<float*>(wsb + g * per);
        xT[g] = reinterpret_cast<float*>(wsb + g * per + pl.ws_wT);
        dyT_ws[g] = reinterpret_cast<float*>(wsb + g * per + pl.ws_wT + pl.ws_xT);
    }

    // dedx fc: dx_g = mask_g * (dy_g . (w_g^T)^T) (and its transpose, rows of N, when asked for)
    if (dx) {
        bool done = false;
        if (pl.dx_tc) {
            const float* const* wt = wT;
            if (!wt) {
                if ((rc = launch_transpose_group(w, ws_wT.data(), batch, out, in, s))) return rc;
                wt = ws_wT.data();
            }
            TcParams p = base_params();
            p.epi = EPI_MASK;
            p.ldd = in;
            p.ldm = in;
            p.lddT = N;
            done = gemm2d_tc_group(dy, out, wt, out, N, in, out, p, nullptr, relu_src, dx, batch, s, &rc, tail_ws,
                                   tail_ws_bytes, dxT);
            if (rc) return rc;
        }
        if (!done) {
            bool transposed = false;
            if (out <= 32 && in % 4 == 0) {
                if ((rc = launch_smallk_dx4(dy, w, relu_src, dx, dxT, batch, N, in, out, s))) return rc;
                transposed = true;
            } else {
                for (int g = 0; g < batch; ++g) {
                    if (out <= 32) {
                        smallk_dx_kernel<<<grid_cap(static_cast<long long>(N) * in), 256, 0, s>>>(
                            dy[g], w[g], relu_src ? relu_src[g] : nullptr, dx[g], N, in, out);
                        if ((rc = check_launch("smallk_dx_kernel"))) return rc;
                    } else {
                        SimtGemm q{N, in, out, dy[g], out, 1, w[g], 1, in, dx[g], in, nullptr,
                                   relu_src ? relu_src[g] : nullptr, in, 1.f, 0, 0, SIMT_MASK};
                        if ((rc = launch_simt_gemm(q, s))) return rc;
                    }
                }
            }
            if (dxT && !transposed &&
                (rc = launch_transpose_group(const_cast<const float* const*>(dx), dxT, batch, N, in, s)))
                return rc;
        }
    }
    // dedw: dw_g = acc*dw_g + alpha * (dy_g^T) . (x_g^T)^T; with x^T followed by a row of
    // ones (xT1) the same GEMM's column `in` is dedb = alpha * sum_i dy_g[i] (+ acc*db_g)
    bool db_done = false;
    {
        bool done = false;
        if (pl.dw_tc) {
            const float* const* bt = xT1;
            if (!bt) {
                if ((rc = launch_transpose_group(x, xT.data(), batch, N, in, s))) return rc;
                bt = xT.data();
            }
            const float* const* at = dyT;
            if (!at) {
                if ((rc = launch_transpose_group(dy, dyT_ws.data(), batch, N, out, s))) return rc;
                at = dyT_ws.data();
            }
            TcParams p = base_params();
            p.epi = EPI_ACCUM;
            p.ldd = in;
            p.alpha = alpha;
            p.accumulate = accumulate;
            const bool with_db = xT1 && db;
            if (with_db) p.vec_col = in;
            done = gemm2d_tc_group(at, N, bt, N, out, with_db ? in + 1 : in, N, p, nullptr, nullptr, dw, batch, s,
                                   &rc, tail_ws, tail_ws_bytes, nullptr, with_db ? db : nullptr);
            if (rc) return rc;
            db_done = done && with_db;
        }
        if (!done) {
            for (int g = 0; g < batch; ++g) {
                SimtGemm q{out, in, N, dy[g], 1, out, x[g], 1, in, dw[g], in, nullptr, nullptr, 0, alpha, accumulate,
                           0, SIMT_ACCUM};
                if ((rc = launch_simt_gemm(q, s))) return rc;
            }
        }
    }
    // dedb
    if (db && !db_done && (rc = launch_colsum_group(dy, db, batch, N, out, alpha, accumulate, s))) return rc;
    return finish_ps();
}

extern "C" int sprint_fc_bwd_batched(const float* const* x, const float* const* xT1, const float* const* w,
                                     const float* const* wT, const float* const* dy, const float* const* dyT,
                                     const float* const* relu_src, float* const* dx, float* const* dxT,
                                     float* const* dw, float* const* db, float alpha, int accumulate, int batch, int N,
                                     int in, int out, void* ws, size_t ws_bytes, sprint_stream_t stream) {
    return fc_bwd_batched_impl(__func__, x, xT1, w, wT, dy, dyT, relu_src, dx, dxT, dw, db, alpha, accumulate, batch,
                               N, in, out, ws, ws_bytes, stream, nullptr);
}

extern "C" int sprint_fc_bwd_update_batched(const float* const* x, const float* const* xT1, const float* const* w,
                                            const float* const* wT, const float* const* dy, const float* const* dyT,
                                            const float* const* relu_src, float* const* dx, float* const* dxT,
                                            float* const* dw, float* const* db, float alpha, int accumulate,
                                            int batch, int N, int in, int out, int opt, const float* w_in,
                                            const float* b_in, float* w_out, float* b_out, float* wT_out,
                                            float* w_state, float* b_state, float eta, float nu_or_eps,
                                            float weight_decay, void* ws, size_t ws_bytes, sprint_stream_t stream) {
    const PsArgs ps{opt, w_in, b_in, w_out, b_out, wT_out, w_state, b_state, eta, nu_or_eps, weight_decay};
    return fc_bwd_batched_impl(__func__, x, xT1, w, wT, dy, dyT, relu_src, dx, dxT, dw, db, alpha, accumulate, batch,
                               N, in, out, ws, ws_bytes, stream, &ps);
}

// ====================================================================== conv
extern "C" size_t sprint_conv_workspace_size(int op, int N, int H, int W, int Cin, int Cout, int pad) {
    if (op < SPRINT_CONV_FWD || op > SPRINT_CONV_DW) return 0;
    if (check_conv_shape(__func__, N, H, W, Cin, Cout, pad) != SPRINT_OK) return 0;
    return plan_conv(op, N, H, W, Cin, Cout, pad, false).ws_total();
}

static int conv_impl_tc(const ConvPlan& pl, const float* act, int act_c, int act_w, int act_h, const CUtensorMap* tb,
                        TcParams p, int ncols, cudaStream_t s, bool* done, float* tail_ws) {
    CUtensorMap ta, td;
    const uint64_t da[4] = {(uint64_t)act_c, (uint64_t)act_w, (uint64_t)act_h, (uint64_t)p.img_n};
    const uint64_t sa[3] = {(uint64_t)act_c * 4, (uint64_t)act_w * act_c * 4, (uint64_t)act_h * act_w * act_c * 4};
    const uint32_t ba[4] = {32, (uint32_t)pl.box.bw, (uint32_t)pl.box.bh, (uint32_t)pl.box.bimg};
    *done = false;
    if (!make_tmap(&ta, act, 4, da, sa, ba)) return SPRINT_OK;
    // the output's 32-row sub-box that one epilogue warp stores (rows are w-fastest pixels)
    const int sbw = pl.box.bw < 32 ? pl.box.bw : 32;
    const int sbh = pl.box.bh < 32 / sbw ? pl.box.bh : 32 / sbw;
    const int sbimg = 32 / (sbw * sbh);
    const uint64_t dd[4] = {(uint64_t)ncols, (uint64_t)p.out_w, (uint64_t)p.out_h, (uint64_t)p.img_n};
    const uint64_t sd[3] = {(uint64_t)p.ldd * 4, (uint64_t)p.out_w * p.ldd * 4, (uint64_t)p.out_h * p.out_w * p.ldd * 4};
    const uint32_t bd[4] = {32, (uint32_t)sbw, (uint32_t)sbh, (uint32_t)sbimg};
    p.store = ST_DIRECT;
    td = ta;
    if ((p.ldd & 3) == 0 && aligned16(p.D) && make_tmap(&td, p.D, 4, dd, sd, bd, false)) p.store = ST_PIX4D;
    p.N = ncols;
    p.num_kt = pl.num_kt;
    p.kt_per_split = pl.num_kt;
    p.bw = pl.box.bw;
    p.bh = pl.box.bh;
    p.bimg = pl.box.bimg;
    p.tiles_w = pl.box.tw;
    p.tiles_h = pl.box.th;
    p.chunks = pl.num_kt / 9;
    *done = true;
    const long long n_tiles = (ncols + pl.tile.bn - 1) / pl.tile.bn;
    const bool tail = pl.gp.tail_splits > 1 && tail_ws;
    if (tail) {
        p.tail_splits = pl.gp.tail_splits;
        p.tail_kt = pl.gp.tail_kt;
        p.tail_start = static_cast<int>(pl.gp.tail_start);
        p.tail_part = tail_ws;
    }
    int rc = launch_tc<ROLE_CONV_IMPL>(pl.tile, ta, *tb, td, p, pl.box.tiles(), n_tiles, 1, s);
    if (rc || !tail) return rc;
    p.tiles_w = pl.box.tw;
    const long long m_units = pl.tile.pair ? (pl.box.tiles() + 1) / 2 : pl.box.tiles();
    return launch_tail_reduce<ROLE_CONV_IMPL>(pl.gp, p, m_units, n_tiles, 1, s);
}

// Persistent CTA pairs of the halo-staged convolution (at most as many as can be resident).
template <int BN>
int launch_halo_bn(const HaloMaps& maps, const TcParams& p, cudaStream_t s) {
    static bool attr_done[64] = {};
    static int slots[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(HALO_THREADS, 1, 1);
    cfg.dynamicSmemBytes = halo_smem_bytes(BN);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(tc_halo_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, halo_smem_bytes(BN)) !=
            cudaSuccess)
            return check_cuda("cudaFuncSetAttribute(tc_halo_kernel)");
        cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, tc_halo_kernel<BN>, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = num_sms() / 2;
        }
        slots[dev] = n;
        attr_done[dev] = true;
    }
    const int pairs = p.num_tiles < slots[dev] ? p.num_tiles : slots[dev];
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.stream = s;
    cudaLaunchKernelEx(&cfg, tc_halo_kernel<BN>, maps, p);
    return check_launch("tc_halo_kernel");
}

// Persistent CTAs of the flipped halo-staged convolution (one per SM at most).
int launch_halo_flip(const HaloMaps& maps, const TcParams& p, cudaStream_t s) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(tc_halo_flip_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, HALO_F_SMEM) !=
            cudaSuccess)
            return check_cuda("cudaFuncSetAttribute(tc_halo_flip_kernel)");
        attr_done[dev] = true;
    }
    const int grid = p.num_tiles < num_sms() ? p.num_tiles : num_sms();
    tc_halo_flip_kernel<<<grid, HALO_THREADS, HALO_F_SMEM, s>>>(maps, p);
    return check_launch("tc_halo_flip_kernel");
}

// The halo-staged implicit GEMM (CTA pairs, BN = ncols = 64 or 128): A = act (NHWC, act_c
// channels) in boxes of (bh + 2) x (bw + 2) pixels around each tile, B through *tb (the map of
// the tap-by-tap implicit GEMM, boxes of BN / 2 rows).
static int conv_halo_tc(const ConvPlan& pl, const float* act, int act_c, int act_w, int act_h, const CUtensorMap* tb,
                        TcParams p, int ncols, cudaStream_t s, bool* done) {
    *done = false;
    CUtensorMap ta;
    const uint64_t da[4] = {(uint64_t)act_c, (uint64_t)act_w, (uint64_t)act_h, (uint64_t)p.img_n};
    const uint64_t sa[3] = {(uint64_t)act_c * 4, (uint64_t)act_w * act_c * 4, (uint64_t)act_h * act_w * act_c * 4};
    const uint32_t ba[4] = {32, (uint32_t)pl.box.bw + 2, (uint32_t)pl.box.bh + 2, 1};
    if (!make_tmap(&ta, act, 4, da, sa, ba)) return SPRINT_OK;
    p.N = ncols;
    p.bw = pl.box.bw;
    p.bh = pl.box.bh;
    p.bimg = 1;
    p.tiles_w = pl.box.tw;
    p.tiles_h = pl.box.th;
    p.chunks = act_c / 32;
    p.num_kt = pl.num_kt;
    p.kt_per_split = pl.num_kt;
    p.store = ST_DIRECT;
    if (pl.hflip) {   // one CTA per tile, all 128 output channels
        SPRINT_REQUIRE(pl.box.tiles() < (1ll << 31), SPRINT_ERR_SHAPE, "conv: %lld halo tiles is too many",
                       pl.box.tiles());
        p.m_tiles = p.num_tiles = static_cast<int>(pl.box.tiles());
        p.n_tiles = p.z_tiles = 1;
        HaloMaps maps;
        maps.a = ta;
        maps.b = *tb;
        maps.d = maps.dt = maps.m = maps.mt = ta;
        *done = true;
        return launch_halo_flip(maps, p, s);
    }
    const long long units = (pl.box.tiles() + 1) / 2, n_tiles = (ncols + pl.tile.bn - 1) / pl.tile.bn;
    SPRINT_REQUIRE(units * n_tiles < (1ll << 31), SPRINT_ERR_SHAPE, "conv: %lld halo tiles is too many",
                   units * n_tiles);
    p.m_tiles = static_cast<int>(units);
    p.n_tiles = static_cast<int>(n_tiles);
    p.z_tiles = 1;
    p.num_tiles = static_cast<int>(units * n_tiles);
    HaloMaps maps;
    maps.a = ta;
    maps.b = *tb;
    maps.d = maps.dt = maps.m = maps.mt = ta;
    p.halo_tma = 0;
    if (pl.tile.bn == 192 && pl.box.bh == 1 && (p.ldd & 3) == 0 && aligned16(p.D) &&
        (!p.mask || ((p.ldm & 3) == 0 && aligned16(p.mask)))) {
        // one-row tiles: each epilogue warp's 32 (or the row's last bw % 32) pixels as TMA boxes of
        // 32 channels, for its stores and its mask block
        const int tw = pl.box.bw % 32;
        const uint64_t dd[4] = {(uint64_t)ncols, (uint64_t)p.out_w, (uint64_t)p.out_h, (uint64_t)p.img_n};
        const uint64_t sd[3] = {(uint64_t)p.ldd * 4, (uint64_t)p.out_w * p.ldd * 4,
                                (uint64_t)p.out_h * p.out_w * p.ldd * 4};
        const uint64_t sm[3] = {(uint64_t)p.ldm * 4, (uint64_t)p.out_w * p.ldm * 4,
                                (uint64_t)p.out_h * p.out_w * p.ldm * 4};
        const uint32_t b32[4] = {32, 32, 1, 1}, btw[4] = {32, (uint32_t)(tw ? tw : 32), 1, 1};
        bool ok = make_tmap(&maps.d, p.D, 4, dd, sd, b32, false) && make_tmap(&maps.dt, p.D, 4, dd, sd, btw, false);
        if (ok && p.mask)
            ok = make_tmap(&maps.m, p.mask, 4, dd, sm, b32, false) && make_tmap(&maps.mt, p.mask, 4, dd, sm, btw, false);
        if (ok) p.halo_tma = 1;
        else maps.d = maps.dt = maps.m = maps.mt = ta;
    }
    *done = true;
    return pl.tile.bn == 192 ? launch_halo_bn<192>(maps, p, s) : launch_halo_bn<128>(maps, p, s);
}

// The halo-staged GEMM factored over the kernel columns (64 outputs): B' = the permuted weights
// [3 * nout][3 * act_c] (fact_weights_kernel), boxes of 96 rows.
static int conv_halo_fact_tc(const ConvPlan& pl, const float* act, int act_c, int act_w, int act_h, int nout,
                             const float* wfact, TcParams p, cudaStream_t s, bool* done) {
    *done = false;
    CUtensorMap tb;
    const uint64_t db[2] = {(uint64_t)3 * act_c, (uint64_t)3 * nout};
    const uint64_t sb[1] = {(uint64_t)3 * act_c * 4};
    const uint32_t bb[2] = {32, pl.tile.b_rows()};
    if (!make_tmap(&tb, wfact, 2, db, sb, bb)) return SPRINT_OK;
    return conv_halo_tc(pl, act, act_c, act_w, act_h, &tb, p, nout, s, done);
}

// The factored implicit GEMM (CONV_FACT, CTA pairs, BN = 192): A = act (NHWC, act_c channels) in
// boxes of 128 pixels of one row, B = the permuted weights [3 * nout][3 * act_c].
static int conv_fact_tc(const ConvPlan& pl, const float* act, int act_c, int act_w, int act_h, int nout,
                        const float* wfact, TcParams p, cudaStream_t s, bool* done) {
    *done = false;
    CUtensorMap ta, tb;
    const uint64_t da[4] = {(uint64_t)act_c, (uint64_t)act_w, (uint64_t)act_h, (uint64_t)p.img_n};
    const uint64_t sa[3] = {(uint64_t)act_c * 4, (uint64_t)act_w * act_c * 4, (uint64_t)act_h * act_w * act_c * 4};
    const uint32_t ba[4] = {32, 32, 1, 1};   // one 32-pixel window
    const int kp = 3 * act_c;
    const uint64_t db[2] = {(uint64_t)kp, (uint64_t)3 * nout};
    const uint64_t sb[1] = {(uint64_t)kp * 4};
    const uint32_t bb[2] = {32, pl.tile.b_rows()};
    if (!make_tmap(&ta, act, 4, da, sa, ba) || !make_tmap(&tb, wfact, 2, db, sb, bb)) return SPRINT_OK;
    p.chunks = act_c / 32;
    p.num_kt = pl.num_kt;
    p.kt_per_split = pl.num_kt;
    p.tiles_w = pl.box.tw;
    // the output through 30-pixel TMA boxes (NHWC, ldd channels per pixel)
    CUtensorMap td = ta;
    const uint64_t dd[4] = {(uint64_t)nout, (uint64_t)p.out_w, (uint64_t)p.out_h, (uint64_t)p.img_n};
    const uint64_t sd[3] = {(uint64_t)p.ldd * 4, (uint64_t)p.out_w * p.ldd * 4, (uint64_t)p.out_h * p.out_w * p.ldd * 4};
    const uint32_t bd[4] = {32, TC_FACT_WIN, 1, 1};
    p.store = ST_DIRECT;
    if ((p.ldd & 3) == 0 && aligned16(p.D) && make_tmap(&td, p.D, 4, dd, sd, bd, false)) p.store = ST_PIX4D;
    TcMaps<1> maps;
    maps.a[0] = ta;
    maps.b[0] = tb;
    maps.d[0] = td;
    const long long tiles = static_cast<long long>(p.img_n) * p.out_h * p.tiles_w;
    const long long units = (tiles + 1) / 2;
    SPRINT_REQUIRE(units < (1ll << 31), SPRINT_ERR_SHAPE, "conv: %lld factored tiles is too many", tiles);
    p.m_tiles = static_cast<int>(units);
    p.n_tiles = 1;
    p.z_tiles = 1;
    p.num_tiles = static_cast<int>(units);
    *done = true;
    return launch_tc_bn<ROLE_CONV_FACT, 192, true, 1>(maps, p, s);
}

extern "C" int sprint_conv_fwd(const float* x, const float* w, const float* b, float* y, int N, int H, int W, int Cin,
                               int Cout, int pad, int relu, void* ws, size_t ws_bytes, sprint_stream_t stream) {
    int rc = check_conv_shape(__func__, N, H, W, Cin, Cout, pad);
    if (rc) return rc;
    SPRINT_NONNULL(x, "x");
    SPRINT_NONNULL(w, "w");
    SPRINT_NONNULL(y, "y");
    SPRINT_ALIGNED(x, "x");
    SPRINT_ALIGNED(w, "w");
    SPRINT_ALIGNED(b, "b");
    SPRINT_ALIGNED(y, "y");
    const ConvPlan pl = plan_conv(SPRINT_CONV_FWD, N, H, W, Cin, Cout, pad, true);
    // the tail-split slabs (last in the workspace) are optional: without room for them the
    // last round is not split
    if ((rc = check_ws(__func__, ws, ws_bytes, pl.ws_total() - pl.ws_tail))) return rc;
    const bool tail_room = pl.ws_tail && ws && ws_bytes >= pl.ws_total();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    if (pl.smallc) return launch_conv_smallc(x, w, b, y, N, H, W, Cin, Cout, pad, relu, s);
    if (pl.rgb) {
        float* wpad = static_cast<float*>(ws);
        pad_cols_kernel<<<(Cout * TC_BK + 255) / 256, 256, 0, s>>>(w, Cout, 9 * Cin, TC_BK, wpad);
        if ((rc = check_launch("pad_cols_kernel"))) return rc;
        const long long P = static_cast<long long>(N) * H * W;
        SPRINT_REQUIRE(P < (1ll << 31) - TC_BM, SPRINT_ERR_SHAPE, "%s: too many output pixels", __func__);
        CUtensorMap tb, td;
        const uint64_t db[2] = {(uint64_t)TC_BK, (uint64_t)Cout}, sb[1] = {(uint64_t)TC_BK * 4};
        const uint32_t bb[2] = {32, 64};
        const uint64_t dd[2] = {(uint64_t)Cout, (uint64_t)P}, sd[1] = {(uint64_t)Cout * 4};
        const uint32_t bd[2] = {32, TC_BM};   // a tile's 128 rows x 32 channels per store
        if (!make_tmap(&tb, wpad, 2, db, sb, bb) || !make_tmap(&td, y, 2, dd, sd, bd, false))
            return fail(SPRINT_ERR_CUDA, "%s: tensor map setup failed", __func__);
        TcParams p = base_params();
        p.M = static_cast<int>(P);
        p.N = Cout;
        p.num_kt = 1;
        p.kt_per_split = 1;
        p.epi = EPI_STORE;
        p.store = ST_2D;
        p.D = y;
        p.ldd = Cout;
        p.bias = b;
        p.relu = relu;
        p.img_n = N;
        p.out_h = H;
        p.out_w = W;
        p.act = x;
        TcMaps<1> maps;
        maps.a[0] = tb;   // (no A map: the producer writes A)
        maps.b[0] = tb;
        maps.d[0] = td;
        p.m_tiles = static_cast<int>((P + TC_BM - 1) / TC_BM);
        p.n_tiles = 1;
        p.z_tiles = 1;
        p.num_tiles = p.m_tiles;
        return launch_tc_bn<ROLE_CONV_RGB, 64, false, 1>(maps, p, s);
    }
    if (pl.fact || (pl.halo && pl.tile.bn == 192)) {
        float* wf = static_cast<float*>(ws);
        fact_weights_kernel<<<grid_cap(9ll * Cin * Cout), 256, 0, s>>>(w, wf, Cin, Cout, 0);
        if ((rc = check_launch("fact_weights_kernel"))) return rc;
        TcParams p = base_params();
        p.img_n = N;
        p.out_h = Ho;
        p.out_w = Wo;
        p.pad = pad;
        p.tap_sign = 1;
        p.epi = EPI_STORE;
        p.D = y;
        p.ldd = Cout;
        p.bias = b;
        p.relu = relu;
        bool done = false;
        rc = pl.halo ? conv_halo_fact_tc(pl, x, Cin, W, H, Cout, wf, p, s, &done)
                     : conv_fact_tc(pl, x, Cin, W, H, Cout, wf, p, s, &done);
        if (rc || done) return rc;
        return fail(SPRINT_ERR_CUDA, "%s: tensor map setup failed", __func__);
    }
    if (pl.tc && pl.im2col) {
        float* col = static_cast<float*>(ws);
        float* wpad = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.ws_col);
        const long long P = static_cast<long long>(N) * Ho * Wo;
        im2col_pad_kernel<<<grid_cap(P * pl.kp), 256, 0, s>>>(x, N, H, W, Cin, pad, pl.kp, col);
        if ((rc = check_launch("im2col_pad_kernel"))) return rc;
        pad_cols_kernel<<<(Cout * pl.kp + 255) / 256, 256, 0, s>>>(w, Cout, 9 * Cin, pl.kp, wpad);
        if ((rc = check_launch("pad_cols_kernel"))) return rc;
        SPRINT_REQUIRE(P < (1ll << 31), SPRINT_ERR_SHAPE, "%s: too many output pixels", __func__);
        TcParams p = base_params();
        p.epi = EPI_STORE;
        p.D = y;
        p.ldd = Cout;
        p.bias = b;
        p.relu = relu;
        if (gemm2d_tc(col, pl.kp, wpad, pl.kp, static_cast<int>(P), Cout, pl.kp, p, s, &rc)) return rc;
        return fail(SPRINT_ERR_CUDA, "%s: tensor map setup failed", __func__);
    }
    if (pl.tc) {
        CUtensorMap tb;
        const uint64_t db[3] = {(uint64_t)Cin, 9, (uint64_t)Cout};
        const uint64_t sb[2] = {(uint64_t)Cin * 4, (uint64_t)9 * Cin * 4};
        const uint32_t bb[3] = {32, 1, pl.tile.b_rows()};
        if (make_tmap(&tb, w, 3, db, sb, bb)) {
            TcParams p = base_params();
            p.img_n = N;
            p.out_h = Ho;
            p.out_w = Wo;
            p.pad = pad;
            p.tap_sign = 1;
            p.b_tap_outer = 0;
            p.epi = EPI_STORE;
            p.D = y;
            p.ldd = Cout;
            p.bias = b;
            p.relu = relu;
            bool done = false;
            float* tail_ws =
                tail_room ? reinterpret_cast<float*>(static_cast<char*>(ws) + pl.ws_total() - pl.ws_tail) : nullptr;
            rc = pl.halo ? conv_halo_tc(pl, x, Cin, W, H, &tb, p, Cout, s, &done)
                         : conv_impl_tc(pl, x, Cin, W, H, &tb, p, Cout, s, &done, tail_ws);
            if (rc || done) return rc;
        }
    }
    const long long total = static_cast<long long>(N) * Ho * Wo * Cout;
    simt_conv_fwd_kernel<<<grid_cap(total), 256, 0, s>>>(x, w, b, y, N, H, W, Cin, Cout, pad, relu);
    return check_launch(__func__);
}

extern "C" int sprint_conv_dX(const float* dy, const float* w, const float* wT, const float* relu_src, float* dx, int N,
                              int H, int W, int Cin, int Cout, int pad, void* ws, size_t ws_bytes,
                              sprint_stream_t stream) {
    int rc = check_conv_shape(__func__, N, H, W, Cin, Cout, pad);
    if (rc) return rc;
    SPRINT_NONNULL(dy, "dy");
    SPRINT_NONNULL(w, "w");
    SPRINT_NONNULL(dx, "dx");
    SPRINT_ALIGNED(dy, "dy");
    SPRINT_ALIGNED(w, "w");
    SPRINT_ALIGNED(wT, "wT");
    SPRINT_ALIGNED(relu_src, "relu_src");
    SPRINT_ALIGNED(dx, "dx");
    const ConvPlan pl = plan_conv(SPRINT_CONV_DX, N, H, W, Cin, Cout, pad, wT != nullptr);
    // the tail-split slabs (last in the workspace) are optional
    if ((rc = check_ws(__func__, ws, ws_bytes, pl.ws_total() - pl.ws_tail))) return rc;
    const bool tail_room = pl.ws_tail && ws && ws_bytes >= pl.ws_total();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    if (pl.fact || (pl.halo && pl.tile.bn == 192)) {
        float* wf = static_cast<float*>(ws);
        fact_weights_kernel<<<grid_cap(9ll * Cin * Cout), 256, 0, s>>>(w, wf, Cin, Cout, 1);
        if ((rc = check_launch("fact_weights_kernel"))) return rc;
        TcParams p = base_params();
        p.img_n = N;
        p.out_h = H;
        p.out_w = W;
        p.pad = pad;
        p.tap_sign = -1;
        p.epi = EPI_MASK;
        p.D = dx;
        p.ldd = Cin;
        p.mask = relu_src;
        p.ldm = Cin;
        bool done = false;
        rc = pl.halo ? conv_halo_fact_tc(pl, dy, Cout, Wo, Ho, Cin, wf, p, s, &done)
                     : conv_fact_tc(pl, dy, Cout, Wo, Ho, Cin, wf, p, s, &done);
        if (rc || done) return rc;
        return fail(SPRINT_ERR_CUDA, "%s: tensor map setup failed", __func__);
    }
    if (pl.tc) {
        const float* wt = wT;
        if (!wt) {
            float* t = static_cast<float*>(ws);
            if ((rc = launch_transpose(w, t, 1, Cout, 9 * Cin, 0, 9ll * Cin, 0, Cout, s))) return rc;
            wt = t;
        }
        CUtensorMap tb;
        const uint64_t db[3] = {(uint64_t)Cout, (uint64_t)Cin, 9};
        const uint64_t sb[2] = {(uint64_t)Cout * 4, (uint64_t)Cin * Cout * 4};
        const uint32_t bb[3] = {32, pl.tile.b_rows(), 1};
        if (make_tmap(&tb, wt, 3, db, sb, bb)) {
            TcParams p = base_params();
            p.img_n = N;
            p.out_h = H;
            p.out_w = W;
            p.pad = pad;
            p.tap_sign = -1;
            p.b_tap_outer = 1;
            p.epi = EPI_MASK;
            p.D = dx;
            p.ldd = Cin;
            p.mask = relu_src;
            p.ldm = Cin;
            bool done = false;
            float* tail_ws =
                tail_room ? reinterpret_cast<float*>(static_cast<char*>(ws) + pl.ws_total() - pl.ws_tail) : nullptr;
            rc = pl.halo ? conv_halo_tc(pl, dy, Cout, Wo, Ho, &tb, p, Cin, s, &done)
                         : conv_impl_tc(pl, dy, Cout, Wo, Ho, &tb, p, Cin, s, &done, tail_ws);
            if (rc || done) return rc;
        }
    }
    const long long total = static_cast<long long>(N) * H * W * Cin;
    simt_conv_dx_kernel<<<grid_cap(total), 256, 0, s>>>(dy, w, relu_src, dx, N, H, W, Cin, Cout, pad);
    return check_launch(__func__);
}

static int conv_dW_impl(const char* fn, const float* x, const float* xT_given, const float* dy, float* dw, float* db,
                        float alpha, int accumulate, int N, int H, int W, int Cin, int Cout, int pad, void* ws,
                        size_t ws_bytes, sprint_stream_t stream);

extern "C" int sprint_conv_dW(const float* x, const float* dy, float* dw, float* db, float alpha, int accumulate,
                              int N, int H, int W, int Cin, int Cout, int pad, void* ws, size_t ws_bytes,
                              sprint_stream_t stream) {
    return conv_dW_impl(__func__, x, nullptr, dy, dw, db, alpha, accumulate, N, H, W, Cin, Cout, pad, ws, ws_bytes,
                        stream);
}

extern "C" size_t sprint_conv_xT_size(int N, int H, int W, int Cin, int Cout, int pad) {
    if (check_conv_shape(__func__, N, H, W, Cin, Cout, pad) != SPRINT_OK) return 0;
    const ConvPlan pl = plan_conv(SPRINT_CONV_DW, N, H, W, Cin, Cout, pad, false);
    return pl.tc && pl.wg_blocked ? pl.ws_xT : 0;
}

extern "C" int sprint_conv_xT(const float* x, float* xT, int N, int H, int W, int Cin, int Cout, int pad,
                              sprint_stream_t stream) {
    int rc = check_conv_shape(__func__, N, H, W, Cin, Cout, pad);
    if (rc) return rc;
    SPRINT_NONNULL(x, "x");
    SPRINT_NONNULL(xT, "xT");
    SPRINT_ALIGNED(x, "x");
    SPRINT_ALIGNED(xT, "xT");
    const ConvPlan pl = plan_conv(SPRINT_CONV_DW, N, H, W, Cin, Cout, pad, false);
    SPRINT_REQUIRE(pl.tc && pl.wg_blocked, SPRINT_ERR_UNSUPPORTED,
                   "%s: this shape's weight gradient reads no blocked copy (N %% 32 != 0 or no tensor-core path)",
                   __func__);
    return launch_transpose(x, xT, H * W, N, Cin, Cin, static_cast<long long>(H) * W * Cin,
                            static_cast<long long>(N) * Cin, 32, static_cast<cudaStream_t>(stream), 32ll * Cin);
}

extern "C" int sprint_conv_dW_xT(const float* x, const float* xT, const float* dy, float* dw, float* db, float alpha,
                                 int accumulate, int N, int H, int W, int Cin, int Cout, int pad, void* ws,
                                 size_t ws_bytes, sprint_stream_t stream) {
    SPRINT_NONNULL(xT, "xT");
    return conv_dW_impl(__func__, x, xT, dy, dw, db, alpha, accumulate, N, H, W, Cin, Cout, pad, ws, ws_bytes,
                        stream);
}

static int conv_dW_impl(const char* fn, const float* x, const float* xT_given, const float* dy, float* dw, float* db,
                        float alpha, int accumulate, int N, int H, int W, int Cin, int Cout, int pad, void* ws,
                        size_t ws_bytes, sprint_stream_t stream) {
    int rc = check_conv_shape(fn, N, H, W, Cin, Cout, pad);
    if (rc) return rc;
    SPRINT_NONNULL(x, "x");
    SPRINT_NONNULL(dy, "dy");
    SPRINT_NONNULL(dw, "dw");
    SPRINT_ALIGNED(x, "x");
    SPRINT_ALIGNED(dy, "dy");
    SPRINT_ALIGNED(dw, "dw");
    SPRINT_ALIGNED(db, "db");
    SPRINT_ALIGNED(xT_given, "xT");
    const ConvPlan pl = plan_conv(SPRINT_CONV_DW, N, H, W, Cin, Cout, pad, false);
    SPRINT_REQUIRE(!xT_given || (pl.tc && pl.wg_blocked), SPRINT_ERR_UNSUPPORTED,
                   "%s: this shape's weight gradient reads no blocked copy of x", fn);
    if ((rc = check_ws(fn, ws, ws_bytes, pl.ws_total()))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Ho = H + 2 * pad - 2, Wo = W + 2 * pad - 2;
    const long long P = static_cast<long long>(N) * Ho * Wo;
    char* wsb = static_cast<char*>(ws);
    float* xT = xT_given ? const_cast<float*>(xT_given) : reinterpret_cast<float*>(wsb);
    float* dyT = reinterpret_cast<float*>(wsb + pl.ws_xT);
    float* part = reinterpret_cast<float*>(wsb + pl.ws_xT + pl.ws_dyT);
    float* csum = reinterpret_cast<float*>(wsb + pl.ws_xT + pl.ws_dyT + pl.ws_partial);
    if (pl.smallc)
        return launch_conv_smallc_dw(x, dy, part, dw, db, alpha, accumulate, N, H, W, Cin, Cout, pad, s);
    bool done = false, db_done = false;
    if (pl.tc) {
        // x [N][H][W][Cin] -> x^T, dy likewise (pixels (h, w, n) = k, n fastest): blocked
        // [H][W*N/32][C][32] when N % 32 == 0, else [C][H][W][N]
        const bool blk = pl.wg_blocked;
        const long long x_db = blk ? static_cast<long long>(N) * Cin : N;
        const long long x_dc = blk ? 32 : static_cast<long long>(H) * W * N;
        const long long y_db = blk ? static_cast<long long>(N) * Cout : N;
        const long long y_dc = blk ? 32 : static_cast<long long>(Ho) * Wo * N;
        if (!xT_given && (rc = launch_transpose(x, xT, H * W, N, Cin, Cin, static_cast<long long>(H) * W * Cin, x_db,
                                                x_dc, s, blk ? 32ll * Cin : 32)))
            return rc;
        // dy -> dy^T, with dedb from the same pass when asked for
        if (db) {
            if ((rc = launch_transpose_colsum(dy, dyT, Ho * Wo, N, Cout, Cout, static_cast<long long>(Ho) * Wo * Cout,
                                              y_db, y_dc, csum, db, alpha, accumulate, s, blk ? 32ll * Cout : 32)))
                return rc;
            db_done = true;
        } else if ((rc = launch_transpose(dy, dyT, Ho * Wo, N, Cout, Cout, static_cast<long long>(Ho) * Wo * Cout, y_db,
                                          y_dc, s, blk ? 32ll * Cout : 32))) {
            return rc;
        }
        CUtensorMap ta, tb;
        // packed taps: one box = one tap's wg_rows channel rows; else BN (or half) channel rows
        const uint32_t b_rows = pl.wg_tpt > 0 ? static_cast<uint32_t>(pl.wg_rows) : pl.tile.b_rows();
        bool maps_ok;
        if (pl.wg_fact) {
            // A = x^T in boxes of 2 rows x Cin = 64 channels, B = dy^T in boxes of 64 and 32 channels
            const uint64_t da[4] = {32, (uint64_t)Cin, (uint64_t)W * N / 32, (uint64_t)H};
            const uint64_t sa[3] = {128, (uint64_t)Cin * 128, (uint64_t)W * N / 32 * Cin * 128};
            const uint64_t dbm[4] = {32, (uint64_t)Cout, (uint64_t)Wo * N / 32, (uint64_t)Ho};
            const uint64_t sbm[3] = {128, (uint64_t)Cout * 128, (uint64_t)Wo * N / 32 * Cout * 128};
            const uint32_t ba[4] = {32, 64, 1, 2}, bb[4] = {32, 64, 1, 1}, bd[4] = {32, 32, 1, 1};
            CUtensorMap tb32;
            maps_ok = make_tmap(&ta, xT, 4, da, sa, ba) && make_tmap(&tb, dyT, 4, dbm, sbm, bb) &&
                      make_tmap(&tb32, dyT, 4, dbm, sbm, bd);
            if (maps_ok) {
                TcParams p = base_params();
                p.M = 2 * TC_BM;
                p.N = 192;
                p.num_kt = pl.num_kt;
                p.kt_per_split = pl.kt_per_split;
                p.splits = pl.splits;
                p.img_n = N;
                p.out_h = Ho;
                p.out_w = Wo;
                p.pad = pad;
                p.tiles_w = pl.box.tw;
                p.tiles_h = pl.box.th;
                p.wg_blocked = 1;
                p.wg_cshift = N / 32;
                p.wg_fact = 1;
                p.wg_slab = wg_fact_slab();
                p.epi = EPI_ACCUM;
                p.store = ST_DIRECT;
                p.partial = part;
                if ((rc = launch_tc<ROLE_CONV_WGRAD>(pl.tile, ta, tb, tb32, p, 2, 1, pl.splits, s))) return rc;
                dw_fact_reduce<<<grid_cap(wg_fact_slab()), 256, 0, s>>>(part, pl.splits, dw, alpha, accumulate);
                if ((rc = check_launch("dw_fact_reduce"))) return rc;
                done = true;
            }
        } else if (blk) {
            const uint64_t da[4] = {32, (uint64_t)Cout, (uint64_t)Wo * N / 32, (uint64_t)Ho};
            const uint64_t sa[3] = {128, (uint64_t)Cout * 128, (uint64_t)Wo * N / 32 * Cout * 128};
            const uint64_t dbm[4] = {32, (uint64_t)Cin, (uint64_t)W * N / 32, (uint64_t)H};
            const uint64_t sbm[3] = {128, (uint64_t)Cin * 128, (uint64_t)W * N / 32 * Cin * 128};
            const uint32_t ba[4] = {32, 128, 1, 1}, bb[4] = {32, b_rows, 1, 1};
            maps_ok = make_tmap(&ta, dyT, 4, da, sa, ba) && make_tmap(&tb, xT, 4, dbm, sbm, bb);
        } else {
            const uint64_t da[3] = {(uint64_t)Wo * N, (uint64_t)Ho, (uint64_t)Cout};
            const uint64_t sa[2] = {(uint64_t)Wo * N * 4, (uint64_t)Ho * Wo * N * 4};
            const uint64_t dbm[3] = {(uint64_t)W * N, (uint64_t)H, (uint64_t)Cin};
            const uint64_t sbm[2] = {(uint64_t)W * N * 4, (uint64_t)H * W * N * 4};
            const uint32_t ba[3] = {32, 1, 128}, bb[3] = {32, 1, b_rows};
            maps_ok = make_tmap(&ta, dyT, 3, da, sa, ba) && make_tmap(&tb, xT, 3, dbm, sbm, bb);
        }
        if (maps_ok && !done) {
            TcParams p = base_params();
            p.M = Cout;
            p.N = Cin;
            p.num_kt = pl.num_kt;
            p.kt_per_split = pl.kt_per_split;
            p.splits = pl.splits;
            p.img_n = N;
            p.out_h = Ho;
            p.out_w = Wo;
            p.pad = pad;
            p.tiles_w = pl.box.tw;
            p.tiles_h = pl.box.th;
            p.wg_blocked = blk ? 1 : 0;
            p.wg_cshift = N / 32;
            p.epi = EPI_ACCUM;
            p.D = dw;
            p.ldd = 9ll * Cin;
            p.alpha = alpha;
            p.accumulate = accumulate;
            p.partial = pl.splits > 1 ? part : nullptr;
            CUtensorMap td = ta;
            p.store = ST_DIRECT;
            if (pl.wg_tpt > 0) {
                // D = [Cout][9 * rows]: straight into dw when rows == Cin and one split, else partials
                const int np = 9 * pl.wg_rows;
                p.wg_tpt = pl.wg_tpt;
                p.wg_rows = pl.wg_rows;
                p.N = np;
                const bool direct = pl.splits == 1 && pl.wg_rows == Cin;
                p.partial = direct ? nullptr : part;
                p.ldd = np;
                if (direct) {
                    const uint64_t dd[2] = {(uint64_t)np, (uint64_t)Cout}, sd[1] = {(uint64_t)np * 4};
                    const uint32_t bd[2] = {32, 32};
                    if ((np & 3) == 0 && make_tmap(&td, dw, 2, dd, sd, bd, false)) p.store = ST_2D;
                } else {
                    const uint64_t dd[3] = {(uint64_t)np, (uint64_t)Cout, (uint64_t)pl.splits};
                    const uint64_t sd[2] = {(uint64_t)np * 4, (uint64_t)Cout * np * 4};
                    const uint32_t bd[3] = {32, 32, 1};
                    if (aligned16(part) && make_tmap(&td, part, 3, dd, sd, bd, false)) p.store = ST_PARTIAL3D;
                }
                if ((rc = launch_tc<ROLE_CONV_WGRAD>(pl.tile, ta, tb, td, p, (Cout + TC_BM - 1) / TC_BM,
                                                     (9 + pl.wg_tpt - 1) / pl.wg_tpt, pl.splits, s)))
                    return rc;
                if (!direct) {
                    dw_packed_reduce<<<grid_cap(9ll * Cout * Cin), 256, 0, s>>>(part, pl.splits, Cout, Cin,
                                                                              pl.wg_rows, dw, alpha, accumulate);
                    if ((rc = check_launch("dw_packed_reduce"))) return rc;
                }
                done = true;
            } else if (pl.splits > 1) {
                const uint64_t dd[3] = {(uint64_t)Cin, (uint64_t)Cout, (uint64_t)9 * pl.splits};
                const uint64_t sd[2] = {(uint64_t)Cin * 4, (uint64_t)Cout * Cin * 4};
                const uint32_t bd[3] = {32, 32, 1};
                if (aligned16(part) && make_tmap(&td, part, 3, dd, sd, bd, false)) p.store = ST_PARTIAL3D;
            } else {
                const uint64_t dd[3] = {(uint64_t)Cin, 9, (uint64_t)Cout};
                const uint64_t sd[2] = {(uint64_t)Cin * 4, (uint64_t)9 * Cin * 4};
                const uint32_t bd[3] = {32, 1, 32};
                if (make_tmap(&td, dw, 3, dd, sd, bd, false)) p.store = ST_WGRAD3D;
            }
            if (!done) {   // one tap per tile: taps and splits in z
                if ((rc = launch_tc<ROLE_CONV_WGRAD>(pl.tile, ta, tb, td, p, (Cout + TC_BM - 1) / TC_BM,
                                                     (Cin + pl.tile.bn - 1) / pl.tile.bn, 9ll * pl.splits, s)))
                    return rc;
                if (pl.splits > 1) {
                    dw_split_reduce<<<grid_cap(9ll * Cout * Cin), 256, 0, s>>>(part, pl.splits, Cout, Cin, dw,
                                                                             alpha, accumulate);
                    if ((rc = check_launch("dw_split_reduce"))) return rc;
                }
                done = true;
            }
        }
    }
    if (!done) {
        SPRINT_REQUIRE(!pl.tc, SPRINT_ERR_CUDA, "%s: tensor map setup failed", __func__);
        const int nchunk = static_cast<int>((P + kDwChunk - 1) / kDwChunk);
        simt_conv_dw_kernel<<<nchunk, 256, 0, s>>>(x, dy, part, N, H, W, Cin, Cout, pad);
        if ((rc = check_launch("simt_conv_dw_kernel"))) return rc;
        const int O = Cout * 9 * Cin;
        colsum_finish_k<<<(O + 255) / 256, 256, 0, s>>>(part, nchunk, O, dw, alpha, accumulate);
        if ((rc = check_launch("colsum_finish_k"))) return rc;
    }
    if (db && !db_done) return launch_colsum(dy, P, Cout, pl.ws_colsum ? csum : nullptr, db, alpha, accumulate, s);
    return SPRINT_OK;
}

// ====================================================================== plan queries
extern "C" int sprint_conv_plan(int op, int N, int H, int W, int Cin, int Cout, int pad, int have_wT, int32_t* out,
                                int n_out) {
    SPRINT_REQUIRE(op >= SPRINT_CONV_FWD && op <= SPRINT_CONV_DW, SPRINT_ERR_INVALID_ARG, "%s: bad op %d", __func__, op);
    int rc = check_conv_shape(__func__, N, H, W, Cin, Cout, pad);
    if (rc) return rc;
    SPRINT_NONNULL(out, "out");
    SPRINT_REQUIRE(n_out >= SPRINT_PLAN_FIELDS, SPRINT_ERR_INVALID_ARG, "%s: out holds %d fields, need %d", __func__,
                   n_out, SPRINT_PLAN_FIELDS);
    const ConvPlan pl = plan_conv(op, N, H, W, Cin, Cout, pad, have_wT != 0);
    for (int i = 0; i < n_out; ++i) out[i] = 0;
    out[0] = pl.smallc ? SPRINT_PATH_SMALLC : (pl.im2col ? SPRINT_PATH_IM2COL : (pl.tc ? SPRINT_PATH_TC : SPRINT_PATH_SIMT));
    out[1] = pl.tile.bn;
    out[2] = pl.tile.pair ? 1 : 0;
    out[3] = pl.splits;
    out[4] = pl.gp.tail_splits;
    out[5] = pl.wg_tpt;
    out[6] = pl.wg_rows;
    out[7] = pl.num_kt;
    out[8] = pl.box.bw;
    out[9] = pl.box.bh;
    out[10] = pl.box.bimg;
    out[11] = pl.wg_blocked ? 1 : 0;
    out[12] = pl.wg_fact ? 1 : 0;
    out[13] = pl.fact ? 1 : 0;
    out[14] = pl.halo ? 1 : 0;
    out[15] = pl.rgb ? 1 : 0;
    out[16] = pl.hflip ? 1 : 0;
    return SPRINT_OK;
}

extern "C" int sprint_gemm_plan(int M, int N, int K, int batch, int allow_tail, int32_t* out, int n_out) {
    SPRINT_REQUIRE(M >= 1 && N >= 1 && K >= 1 && batch >= 1, SPRINT_ERR_SHAPE, "%s: need M, N, K, batch >= 1", __func__);
    SPRINT_NONNULL(out, "out");
    SPRINT_REQUIRE(n_out >= SPRINT_PLAN_FIELDS, SPRINT_ERR_INVALID_ARG, "%s: out holds %d fields, need %d", __func__,
                   n_out, SPRINT_PLAN_FIELDS);
    const long long m_tiles = (M + TC_BM - 1) / TC_BM;
    const int per_launch = batch < kMaxGroup ? batch : kMaxGroup;
    const GemmPlan plan =
        plan_gemm(m_tiles, N, per_launch, N >= 256 ? 256 : (N >= 128 ? 128 : 64), (K + TC_BK - 1) / TC_BK, allow_tail != 0);
    for (int i = 0; i < n_out; ++i) out[i] = 0;
    out[0] = SPRINT_PATH_TC;
    out[1] = plan.tile.bn;
    out[2] = plan.tile.pair ? 1 : 0;
    out[3] = 1;
    out[4] = plan.tail_splits;
    out[7] = (K + TC_BK - 1) / TC_BK;
    return SPRINT_OK;
}
