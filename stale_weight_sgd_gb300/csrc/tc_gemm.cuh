// tcgen05 TF32 GEMM engine for the contractions of the worker step.
//
// Persistent kernel: gridDim.x CTAs (at most one per SM) walk a static list of
// 128 x BN output tiles (m fastest, so CTAs running together share the B
// panel in L2). Within a CTA:
//   warp 4   : TMA producer (one lane) — fills a STAGES-deep ring of shared-
//              memory stages, each one or two k-tiles of 128 B (32 fp32) along
//              k, 128-byte swizzled; the ring runs on across tiles;
//   warp 5   : allocates two TMEM accumulators (BN fp32 columns each) and issues
//              tcgen05.mma.kind::tf32 (M=128, N=BN, K=8) from one lane, tile
//              after tile, alternating accumulators; tcgen05.commit frees a
//              stage once its MMAs are done and hands a finished accumulator
//              to the epilogue;
//   warps 0-3: epilogue — tcgen05.ld the accumulator (warp w owns TMEM lanes
//              32w..32w+31 = tile rows), release it to the MMA warp, apply
//              bias/ReLU, the ReLU mask of the backward pass or the GradBuf
//              scale, stage each 32 x 32 chunk in 128B-swizzled shared memory
//              and write it with a TMA store (or a TMA add-reduction for the
//              GradBuf accumulate); ragged edges are clipped by TMA. Outputs TMA
//              cannot describe (row pitch not a multiple of 16 bytes) are
//              written by the threads directly instead.
// So the epilogue of tile i overlaps the MMAs of tile i+1. The hand-back is a
// relaxed arrive: a release would first wait for the warp's earlier direct
// stores (transposed copies, vector columns) to become visible.
//
// CTA pairs (PAIR = true, clusters of two): a work unit is two vertically
// adjacent tiles (m-tiles 2u and 2u+1) computed by one tcgen05.mma of M = 256
// (cta_group::2) that the even CTA issues. Each CTA loads its own 128 rows of A
// and half of the BN rows of B, so a pair moves 3/4 of the operand bytes two
// single CTAs would for the same FLOPs; both CTAs' loads complete on the even
// CTA's stage barrier, commits free the stage in both CTAs, and each CTA's
// epilogue drains its own TMEM (rows 0-127 of the pair tile in the even CTA,
// 128-255 in the odd one) and hands it back to the even CTA's MMA thread.
//
// Both operands are K-major: the TF32 kind of tcgen05.mma reads no MN-major
// operand on this part, so transposed operands are formed in global memory by
// the callers (gemm.cu). Every wait is bounded: one that gives up sets a bit
// in the device status word and the CTA finishes without hanging.
//
// Roles (the SGEMM roles of the SPRINT report, Sec. 3.3):
//   GEMM_2D   : A [M][K], B [N][K] row-major (fc, dedx fc with B = w^T,
//               dedw fc with A = dy^T and B = x^T)
//   CONV_IMPL : implicit-GEMM convolution — A = 128 NHWC pixels (4-D box,
//               shifted by the tap, halo zero-filled by TMA), B = the tap's
//               weight slice (3-D box). Forward: A = x, B = w[co][tap][ci];
//               dedx conv: A = dy at the mirrored tap, B = w^T[tap][ci][co].
//   CONV_FACT : forward or input gradient of a layer whose output has 64
//               channels, factored over the kernel columns (CTA pairs, BN =
//               192): D'[q][(dw, c)] = sum over (dh, k) of A[q + s*(dh-1, 0)][k]
//               * B'[(dw, c)][(dh, k)], with q = four windows of 32 consecutive
//               pixels of one image row (each window one pixel wider on both
//               sides than its 30 outputs), A = x (s = +1) or dy (s = -1) and B'
//               the weights permuted by the host; the epilogue adds the three
//               column blocks of neighbouring rows within the warp's window:
//               out[q] = D'[q - s][dw 0] + D'[q][dw 1] + D'[q + s][dw 2].
//   CONV_RGB  : forward of a layer with 3 input channels (the RGB layer, pad 1):
//               one k-tile per 128-pixel tile, A = the tile's im2col rows
//               ((dh * 3 + dw) * 3 + c, zero past 27) written into shared memory
//               from x (act, NHWC) by four more warps (6-9, one row per lane),
//               B = the weights padded to 32 columns (TMA, warp 4); the stage's
//               barrier takes the TMA bytes and one arrival per im2col warp; the
//               epilogue writes y [pixels][64] as two TMA boxes of 128 rows x 32
//               channels per tile (double-buffered), the four warps' rows together.
//   CONV_WGRAD: dedw conv, per tap: A = dy^T, B = x^T shifted by the tap; a
//               k-tile is 32 consecutive (w, n) positions of one row, n fastest,
//               so the tap's w-shift is N positions. The copies are either
//               [C][H][W][N] or, when N % 32 == 0, blocked [H][W*N/32][C][32]:
//               there a k-tile of C channel rows is one contiguous C x 128-byte
//               block (the first form spreads its rows H*W*N*4 bytes apart, a
//               page or more each on wide images) and the w-shift is N/32 whole
//               blocks. Every TMA box here is 128 B wide along its inner
//               dimension, the 128-byte swizzle span.
#pragma once

#include "common.cuh"

namespace sprint {

enum Role : int { ROLE_GEMM_2D = 0, ROLE_CONV_IMPL = 1, ROLE_CONV_WGRAD = 2, ROLE_CONV_FACT = 3, ROLE_CONV_RGB = 4 };
enum Epi : int { EPI_STORE = 0, EPI_MASK = 1, EPI_ACCUM = 2 };
// how the epilogue writes: direct stores, or TMA through a store map of shape
enum Store : int { ST_DIRECT = 0, ST_2D = 1, ST_PIX4D = 2, ST_WGRAD3D = 3, ST_PARTIAL3D = 4 };

constexpr int TC_BM = 128;
// CONV_FACT: each epilogue warp's 32 rows are a window of 32 consecutive
// pixels of which the middle 30 are outputs (its first and last rows are the
// halo its neighbours need), so a 128-row tile yields 120 outputs
constexpr int TC_FACT_WIN = 30;
constexpr int TC_FACT_OUT = 4 * TC_FACT_WIN;
constexpr int TC_BK = 32;                      // fp32 elements per 128-byte swizzle row
constexpr int TC_THREADS = 192;
constexpr int TC_A_STAGE = TC_BM * TC_BK * 4;  // 16 KB
constexpr int TC_STAGING = 4 * 4096;           // one 32 x 32 fp32 staging chunk per epilogue warp

// B rows one CTA holds per k-tile (a pair splits the BN rows between its CTAs)
__host__ __device__ constexpr int tc_b_rows(int bn, bool pair) { return pair ? bn / 2 : bn; }
__host__ __device__ constexpr int tc_b_stage(int bn, bool pair) { return tc_b_rows(bn, pair) * TC_BK * 4; }
constexpr int TC_RING_BYTES = 232448 - 1024 - 4 * 4096 - 1024;   // shared memory left for the operand ring
// k-tiles per pipeline stage. Every stage hand-off (full barrier, MMA batch,
// commit) costs a roughly fixed ~100 cycles, which narrow tiles cannot hide
// behind their MMAs, so they take two k-tiles per stage as long as the ring
// still holds at least four stages (measured: +20-30% for pair tiles of width
// <= 160 and single tiles of width 64; wide tiles lose more from the shorter
// ring than they gain).
__host__ __device__ constexpr int tc_ks(int bn, bool pair) {
    return TC_RING_BYTES / (2 * (TC_A_STAGE + tc_b_stage(bn, pair))) >= 4 ? 2 : 1;
}
// as many stages as fit next to the staging buffers in 227 KB of shared memory (at most 8)
__host__ __device__ constexpr int tc_stages(int bn, bool pair) {
    return TC_RING_BYTES / (tc_ks(bn, pair) * (TC_A_STAGE + tc_b_stage(bn, pair))) > 8
               ? 8
               : TC_RING_BYTES / (tc_ks(bn, pair) * (TC_A_STAGE + tc_b_stage(bn, pair)));
}
__host__ __device__ constexpr int tc_tmem_cols(int bn) { return bn <= 32 ? 64 : (bn <= 64 ? 128 : (bn <= 128 ? 256 : 512)); }
__host__ __device__ constexpr int tc_smem_bytes(int bn, bool pair) {
    return 1024 /* alignment slack */ +
           tc_stages(bn, pair) * tc_ks(bn, pair) * (TC_A_STAGE + tc_b_stage(bn, pair)) + TC_STAGING +
           256 /* barriers */;
}

// CONV_RGB (one k-tile per tile) takes stages of one k-tile and four staging buffers per epilogue
// warp, so that a warp does not wait for its last TMA store to read its buffer; every other role
// the shapes above.
template <int ROLE>
__host__ __device__ constexpr int tc_nstg() { return ROLE == ROLE_CONV_RGB ? 4 : 1; }
template <int ROLE>
__host__ __device__ constexpr int tc_ks_r(int bn, bool pair) { return ROLE == ROLE_CONV_RGB ? 1 : tc_ks(bn, pair); }
template <int ROLE>
__host__ __device__ constexpr int tc_stages_r(int bn, bool pair) {
    return ROLE == ROLE_CONV_RGB ? 4 : tc_stages(bn, pair);
}
template <int ROLE>
__host__ __device__ constexpr int tc_smem_bytes_r(int bn, bool pair) {
    return ROLE == ROLE_CONV_RGB ? 1024 + tc_stages_r<ROLE>(bn, pair) * tc_ks_r<ROLE>(bn, pair) *
                                              (TC_A_STAGE + tc_b_stage(bn, pair)) +
                                       tc_nstg<ROLE>() * TC_STAGING + 256
                                 : tc_smem_bytes(bn, pair);
}

// Up to TC_MAX_GROUP independent GEMMs of one shape in one launch (the work
// units of problem g have z = g): one tensor-map triple per problem.
constexpr int TC_MAX_GROUP = kMaxGroup;
template <int G>
struct TcMaps {
    CUtensorMap a[G], b[G], d[G];
};

struct TcParams {
    int M, N;            // GEMM_2D / CONV_WGRAD: output rows, columns; CONV_IMPL: N = columns
    int m_tiles, n_tiles, z_tiles, num_tiles;  // work units: m fastest, then n, then z (a pair's
                                               // unit covers m-tiles 2m and 2m+1)
    int num_kt;          // k-tiles in the full reduction
    int kt_per_split;    // k-tiles per split
    int splits;          // CONV_WGRAD: z = tap * splits + split
    // convolution geometry: pixel boxes (bw x bh x bimg) tile the output grid
    int img_n, out_h, out_w, pad;
    int bw, bh, bimg, tiles_w, tiles_h;
    int chunks;          // CONV_IMPL: 32-channel chunks per tap
    int tap_sign;        // CONV_IMPL: +1 forward (x[p + tap - pad]), -1 dedx (dy[p - tap + pad])
    int b_tap_outer;     // CONV_IMPL: B map dims {k, n, 9} (1) or {k, 9, n} (0)
    // epilogue
    int epi;
    int store;           // Store
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
    // tail split (GEMM_2D): units from tail_start on are the last, partial
    // round's tiles, each cut into tail_splits k-ranges of tail_kt k-tiles; their
    // raw accumulators go to tail_part (one TM x BN fp32 slab per unit, TM = 256
    // for a pair, 128 otherwise) and tc_tail_reduce finishes them
    int tail_start, tail_splits, tail_kt;
    float* tail_part;
    // CONV_WGRAD with taps packed along N (wg_tpt > 0): an n-tile holds wg_tpt
    // taps of wg_rows channel rows each (wg_rows % 8 == 0: every tap's slice
    // starts on a 1024-byte swizzle atom; rows past Cin are TMA zero fill), so
    // D[co][tap * wg_rows + ci]; z is the k split only. wg_tpt == 0: one tap per
    // n-tile column range, taps and splits in z.
    int wg_tpt, wg_rows;
    // CONV_WGRAD operand layout: 0 = [C][H][W][N] (maps {W*N, H, C}); 1 = blocked
    // [H][W*N/32][C][32] (maps {32, C, W*N/32, H}: a k-tile box is C rows of 128
    // contiguous bytes, and the tap's w-shift of N elements is wg_cshift = N/32
    // whole blocks)
    int wg_blocked, wg_cshift;
    // CONV_WGRAD factored over the kernel rows and columns (wg_fact = 1; CTA
    // pairs, BN = 192, Cin = Cout = 64, pad 1, blocked copies): the identity
    // dW[co][dh][dw][ci] = sum_q dy[q - (0, dw-1)][co] x[q + (dh-1, 0)][ci]
    // makes D = [(dh, ci)] x [(dw, co)], A = x^T shifted by dh (the even CTA's
    // rows dh 0 and 1, the odd CTA's dh 2), B = dy^T shifted by -(dw-1): all nine
    // taps from 2 + 4 boxes per k-tile, no half-empty tile for Cout = 64 (the odd
    // CTA's A rows 64-127, x^T two rows down, are never stored). maps.a holds
    // x^T boxes of 2 rows x 64 channels, maps.b dy^T boxes of 64 channels and
    // maps.d of 32. Each split writes one slab of wg_slab floats (dW in its
    // [co][tap][ci] layout) at partial + split * wg_slab.
    int wg_fact;
    long long wg_slab;
    // grouped launches: per-problem bias, mask and output (direct stores)
    const float* g_bias[TC_MAX_GROUP];
    const float* g_mask[TC_MAX_GROUP];
    float* g_D[TC_MAX_GROUP];
    // grouped launches, direct stores by the thread that owns the row:
    //  g_DT[z] (optional): a transposed copy of the output, DT[n * lddT + m]
    //  (EPI_STORE, EPI_MASK);
    //  vec_col >= 0 (EPI_ACCUM): GEMM column vec_col is not part of D (which
    //  holds the vec_col columns before it) but lands in g_vec[z][m], with the
    //  same alpha / accumulate epilogue (a column of ones appended to B turns
    //  it into the row sums of A)
    int vec_col;
    long long lddT;
    float* g_DT[TC_MAX_GROUP];
    float* g_vec[TC_MAX_GROUP];
    // unit order m, then z, then n (grouped problems that share B run their
    // units of one n-tile together, so each B tile comes from HBM once);
    // 0: m, then n, then z
    int z_mid;
    // CONV_RGB: the layer input x [img_n][out_h][out_w][3]
    const float* act;
    // halo-staged kernel, factored tiles of one output row: each epilogue warp loads its mask block
    // and stores its outputs by TMA (maps d / m: 32-pixel boxes, dt / mt: the row's last bw % 32)
    int halo_tma;
};

#if defined(__CUDACC__)

struct TileCoord {
    int mt, nt, z;
    int tail;   // index of a tail-split unit (-1: a whole tile)
    int split;  // its k-range
};

__host__ __device__ __forceinline__ TileCoord tile_coord(int t, const TcParams& p) {
    TileCoord c;
    c.tail = -1;
    c.split = 0;
    int tt = t;
    if (p.tail_splits > 1 && t >= p.tail_start) {
        const int u = t - p.tail_start;
        tt = p.tail_start + u / p.tail_splits;
        c.tail = u;
        c.split = u % p.tail_splits;
    }
    c.mt = tt % p.m_tiles;
    const int r = tt / p.m_tiles;
    if (p.z_mid) {
        c.z = r % p.z_tiles;
        c.nt = r / p.z_tiles;
    } else {
        c.nt = r % p.n_tiles;
        c.z = r / p.n_tiles;
    }
    return c;
}

// CONV_FACT tile mt: image n, row h, first output pixel w0 (tiles_w tiles of
// TC_FACT_OUT outputs per image row); n >= img_n past the last tile
__host__ __device__ __forceinline__ void fact_tile(const TcParams& p, int mt, int& n, int& h, int& w0) {
    const int per_img = p.out_h * p.tiles_w;
    n = mt / per_img;
    const int rem = mt % per_img;
    h = rem / p.tiles_w;
    w0 = (rem % p.tiles_w) * TC_FACT_OUT;
}

// CONV_RGB adds warps 6-9, which write the im2col rows
template <int ROLE>
__host__ __device__ constexpr int tc_threads() { return ROLE == ROLE_CONV_RGB ? TC_THREADS + 128 : TC_THREADS; }

template <int ROLE, int BN, bool PAIR, int G>
__global__ void __launch_bounds__(tc_threads<ROLE>(), 1)
    tc_gemm_kernel(const __grid_constant__ TcMaps<G> maps, const TcParams p) {
    static_assert(G == 1 || ROLE == ROLE_GEMM_2D, "only plain GEMMs are grouped");
    constexpr int STAGES = tc_stages_r<ROLE>(BN, PAIR);
    constexpr int KS = tc_ks_r<ROLE>(BN, PAIR);  // k-tiles per stage
    constexpr int NSTG = tc_nstg<ROLE>();        // staging buffers per epilogue warp
    constexpr int B_ROWS = tc_b_rows(BN, PAIR);
    constexpr int B_STAGE = tc_b_stage(BN, PAIR);  // one k-tile of B
    constexpr uint32_t IDESC = idesc_tf32(BN, false, false, PAIR ? 256 : 128);
    constexpr uint32_t TMEM_COLS = tc_tmem_cols(BN);
    // bytes of one k-tile on the barrier the MMA thread waits on (both CTAs' loads for a pair)
    constexpr uint32_t KTILE_BYTES = (TC_A_STAGE + B_STAGE) * (PAIR ? 2 : 1);
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN must be a multiple of 32 in [32, 256]");
    static_assert(!PAIR || BN >= 64, "a pair splits BN into two halves of at least 32 rows");
    static_assert(tc_smem_bytes_r<ROLE>(BN, PAIR) <= 232448, "shared memory budget exceeded");
    constexpr uint32_t ACC_STRIDE = TMEM_COLS / 2;   // second accumulator at a power-of-two column offset

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * KS * TC_A_STAGE;
    uint8_t* sStage = sB + STAGES * KS * B_STAGE;   // 4 x NSTG x 4 KB epilogue staging, 1024-aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(sStage + NSTG * TC_STAGING);
    uint64_t* empty = full + STAGES;
    uint64_t* tmem_full = empty + STAGES;     // [2]
    uint64_t* tmem_empty = tmem_full + 2;     // [2]
    uint64_t* mma_done = tmem_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // position in the pair (0 = the CTA that issues the MMAs); work unit walk
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const int unit0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (warp == 4 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], ROLE == ROLE_CONV_RGB ? 5 : 1);   // CONV_RGB: + one arrival per im2col warp
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tmem_full[b], 1);
            mbar_init(&tmem_empty[b], PAIR ? 8 : 4);   // one arrival per epilogue warp (of both CTAs)
        }
        mbar_init(mma_done, 1);
        fence_mbar_init();
        for (int g = 0; g < G && g < p.z_tiles; ++g) {
            tma_prefetch_desc(&maps.a[g]);
            tma_prefetch_desc(&maps.b[g]);
            if (p.store != ST_DIRECT || p.wg_fact) tma_prefetch_desc(&maps.d[g]);
        }
    }
    if (warp == 5) {
        if constexpr (PAIR) {
            tmem_alloc_pair(tmem_slot, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();   // the peer's barriers are initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // this CTA's tile of work unit t
    auto own_coord = [&](int t) {
        TileCoord c = tile_coord(t, p);
        if constexpr (PAIR) c.mt = 2 * c.mt + static_cast<int>(rank);
        return c;
    };

    // per-tile k range (split-K over z for the weight gradient)
    auto k_range = [&](const TileCoord& tc, int& kt0, int& nkt, int& tap) {
        tap = 0;
        if (tc.tail >= 0) {
            kt0 = tc.split * p.tail_kt;
            const int kt1 = kt0 + p.tail_kt < p.num_kt ? kt0 + p.tail_kt : p.num_kt;
            nkt = kt1 > kt0 ? kt1 - kt0 : 0;
            return;
        }
        int split = G > 1 ? 0 : tc.z;   // grouped: z is the problem, not a k split
        tap = 0;
        if constexpr (ROLE == ROLE_CONV_WGRAD) {
            if (p.wg_tpt == 0 && !p.wg_fact) {
                tap = tc.z / p.splits;
                split = tc.z % p.splits;
            }
            // interleaved splits: split s takes k-tiles s, s + splits, ... so the CTAs running
            // together read one narrow k window (shared through L2, rows swept in order)
            // instead of `splits` far-apart streams of the [C][H][W][N] copies
            kt0 = split;
            nkt = split < p.num_kt ? (p.num_kt - split + p.splits - 1) / p.splits : 0;
            return;
        }
        kt0 = split * p.kt_per_split;
        int kt1 = kt0 + p.kt_per_split;
        if (kt1 > p.num_kt) kt1 = p.num_kt;
        nkt = kt1 > kt0 ? kt1 - kt0 : 0;
    };

    if (warp == 4) {
        // ---------------------------------------------------------------- TMA producer
        if constexpr (ROLE == ROLE_CONV_RGB) {
            // the weights of each tile's stage (warps 6-9 write its im2col rows)
            if (lane == 0) {
                uint32_t it = 0;
                for (int t = unit0; t < p.num_tiles; t += units, ++it) {
                    const uint32_t s = it % STAGES;
                    if (!mbar_wait_bounded(&empty[s], ((it / STAGES) & 1) ^ 1, p.status, DEV_FLAG_WAIT_PRODUCER)) break;
                    mbar_arrive_expect_tx(&full[s], B_STAGE);
                    tma_load_2d(sB + s * KS * B_STAGE, &maps.b[0], 0, 0, &full[s]);
                }
                // every weight copy issued above has landed before the CTA may exit
                for (uint32_t k = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u; k < it; ++k)
                    if (!mbar_wait_bounded(&full[k % STAGES], (k / STAGES) & 1, p.status, DEV_FLAG_WAIT_PRODUCER))
                        break;
            }
        } else if (lane == 0) {
            uint32_t it = 0;
            bool alive = true;
            for (int t = unit0; t < p.num_tiles && alive; t += units) {
                const TileCoord tc = own_coord(t);
                int kt0, nkt, tap;
                k_range(tc, kt0, nkt, tap);
                const CUtensorMap* mA = &maps.a[G > 1 ? tc.z : 0];
                const CUtensorMap* mB = &maps.b[G > 1 ? tc.z : 0];
                // B rows this CTA loads: all BN, or its half of them in a pair
                const int n0 = tc.nt * BN + static_cast<int>(rank) * B_ROWS, m0 = tc.mt * TC_BM;
                int pw0 = 0, ph0 = 0, pn0 = 0;
                if constexpr (ROLE == ROLE_CONV_IMPL) {
                    pw0 = (tc.mt % p.tiles_w) * p.bw;
                    ph0 = ((tc.mt / p.tiles_w) % p.tiles_h) * p.bh;
                    pn0 = (tc.mt / (p.tiles_w * p.tiles_h)) * p.bimg;
                } else if constexpr (ROLE == ROLE_CONV_FACT) {
                    fact_tile(p, tc.mt, pn0, ph0, pw0);
                }
                for (int i = 0; i < nkt; i += KS, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1, p.status, DEV_FLAG_WAIT_PRODUCER)) {
                        alive = false;
                        break;
                    }
                    const int nq = nkt - i < KS ? nkt - i : KS;   // k-tiles in this stage
                    uint32_t ktile_bytes = KTILE_BYTES;
                    if constexpr (ROLE == ROLE_CONV_WGRAD) {
                        if (p.wg_fact) {   // x^T: one 128-row box per CTA; dy^T: 64 + 32 rows per CTA
                            ktile_bytes = 2u * 128u * 128u + 2u * 96u * 128u;
                        } else if (p.wg_tpt > 0) {   // A boxes of both CTAs + the taps that exist in this n-tile
                            const int per = PAIR ? p.wg_tpt / 2 : p.wg_tpt;
                            int taps = 0;
                            for (int rk = 0; rk < (PAIR ? 2 : 1); ++rk) {
                                const int first = tc.nt * p.wg_tpt + rk * per;
                                taps += first >= 9 ? 0 : (9 - first < per ? 9 - first : per);
                            }
                            ktile_bytes = (PAIR ? 2u : 1u) * TC_A_STAGE + static_cast<uint32_t>(taps * p.wg_rows) * 128u;
                        }
                    }
                    if (rank == 0) mbar_arrive_expect_tx(&full[s], nq * ktile_bytes);
                    for (int q = 0; q < nq; ++q) {
                        // the k-tile of this stage slot (interleaved splits for the weight gradient)
                        const int kt = ROLE == ROLE_CONV_WGRAD ? kt0 + (i + q) * p.splits : kt0 + i + q;
                        uint8_t* a_dst = sA + (s * KS + q) * TC_A_STAGE;
                        uint8_t* b_dst = sB + (s * KS + q) * B_STAGE;
                        if constexpr (PAIR) {
                            // both CTAs' copies complete on the even CTA's barrier
                            const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);
                            if constexpr (ROLE == ROLE_GEMM_2D) {
                                tma_load_2d_pair(a_dst, mA, kt * TC_BK, m0, bar);
                                tma_load_2d_pair(b_dst, mB, kt * TC_BK, n0, bar);
                            } else if constexpr (ROLE == ROLE_CONV_IMPL) {
                                const int tp = kt / p.chunks;
                                const int c0 = (kt % p.chunks) * TC_BK;
                                const int dh = (tp / 3 - p.pad) * p.tap_sign, dw = (tp % 3 - p.pad) * p.tap_sign;
                                tma_load_4d_pair(a_dst, mA, c0, pw0 + dw, ph0 + dh, pn0, bar);
                                if (p.b_tap_outer)
                                    tma_load_3d_pair(b_dst, mB, c0, n0, tp, bar);
                                else
                                    tma_load_3d_pair(b_dst, mB, c0, tp, n0, bar);
                            } else if constexpr (ROLE == ROLE_CONV_FACT) {
                                // A: the four 32-pixel windows of the row shifted by the kernel row (zero fill
                                // outside the image, and past the last tile); B': the permuted weights, k =
                                // (dh, channel)
                                const int dh = kt / p.chunks;
                                const int c0 = (kt % p.chunks) * TC_BK;
#pragma unroll
                                for (int wi = 0; wi < 4; ++wi)
                                    tma_load_4d_pair(a_dst + wi * 32 * 128, mA, c0, pw0 + wi * TC_FACT_WIN - 1,
                                                     ph0 + p.tap_sign * (dh - 1), pn0, bar);
                                tma_load_2d_pair(b_dst, mB, kt * TC_BK, n0, bar);
                            } else if (p.wg_fact) {   // factored: A = x^T rows (dh, ci), B = dy^T rows (dw, co)
                                const int h = kt / p.tiles_w;
                                const int ck = kt % p.tiles_w;
                                // A: the 2-row box of x^T rows h - 1, h (even CTA) or h + 1, h + 2 (odd CTA,
                                // whose second half, rows 64-127, is never stored)
                                tma_load_4d_pair(a_dst, mA, 0, 0, ck, h - 1 + 2 * static_cast<int>(rank), bar);
                                // B rows (dw, co): even CTA dw 0 (a 64-row box of maps.b) and dw 1 co 0-31, odd
                                // CTA dw 1 co 32-63 and dw 2 (32-row boxes of maps.d)
                                const CUtensorMap* mB32 = &maps.d[0];
                                if (rank == 0) {
                                    tma_load_4d_pair(b_dst, mB, 0, 0, ck + p.wg_cshift, h, bar);
                                    tma_load_4d_pair(b_dst + 64 * 128, mB32, 0, 0, ck, h, bar);
                                } else {
                                    tma_load_4d_pair(b_dst, mB32, 0, 32, ck, h, bar);
                                    tma_load_4d_pair(b_dst + 32 * 128, mB, 0, 0, ck - p.wg_cshift, h, bar);
                                }
                            } else if (p.wg_blocked) {   // blocked [H][W*N/32][C][32] copies
                                const int h = kt / p.tiles_w;
                                const int ck = kt % p.tiles_w;
                                tma_load_4d_pair(a_dst, mA, 0, m0, ck, h, bar);
                                if (p.wg_tpt > 0) {
                                    const int per = p.wg_tpt / 2, first = tc.nt * p.wg_tpt + static_cast<int>(rank) * per;
                                    for (int j = 0; j < per && first + j < 9; ++j) {
                                        const int tp = first + j;
                                        tma_load_4d_pair(b_dst + j * p.wg_rows * 128, mB, 0, 0,
                                                         ck + (tp % 3 - p.pad) * p.wg_cshift, h + tp / 3 - p.pad, bar);
                                    }
                                } else {
                                    tma_load_4d_pair(b_dst, mB, 0, n0, ck + (tap % 3 - p.pad) * p.wg_cshift,
                                                     h + tap / 3 - p.pad, bar);
                                }
                            } else {
                                const int h = kt / p.tiles_w;
                                const int c0 = (kt % p.tiles_w) * TC_BK;
                                tma_load_3d_pair(a_dst, mA, c0, h, m0, bar);
                                if (p.wg_tpt > 0) {
                                    const int per = p.wg_tpt / 2, first = tc.nt * p.wg_tpt + static_cast<int>(rank) * per;
                                    for (int j = 0; j < per && first + j < 9; ++j) {
                                        const int tp = first + j;
                                        tma_load_3d_pair(b_dst + j * p.wg_rows * 128, mB, c0 + (tp % 3 - p.pad) * p.img_n,
                                                         h + tp / 3 - p.pad, 0, bar);
                                    }
                                } else {
                                    tma_load_3d_pair(b_dst, mB, c0 + (tap % 3 - p.pad) * p.img_n, h + tap / 3 - p.pad,
                                                     n0, bar);
                                }
                            }
                        } else if constexpr (ROLE == ROLE_GEMM_2D) {
                            tma_load_2d(a_dst, mA, kt * TC_BK, m0, &full[s]);
                            tma_load_2d(b_dst, mB, kt * TC_BK, n0, &full[s]);
                        } else if constexpr (ROLE == ROLE_CONV_IMPL) {
                            const int tp = kt / p.chunks;
                            const int c0 = (kt % p.chunks) * TC_BK;
                            const int dh = (tp / 3 - p.pad) * p.tap_sign, dw = (tp % 3 - p.pad) * p.tap_sign;
                            tma_load_4d(a_dst, mA, c0, pw0 + dw, ph0 + dh, pn0, &full[s]);
                            if (p.b_tap_outer)
                                tma_load_3d(b_dst, mB, c0, n0, tp, &full[s]);
                            else
                                tma_load_3d(b_dst, mB, c0, tp, n0, &full[s]);
                        } else if (p.wg_blocked) {  // CONV_WGRAD, blocked: dy^T {32, Cout, Wo*N/32, Ho}, x^T {32, Cin, W*N/32, H}
                            const int h = kt / p.tiles_w;
                            const int ck = kt % p.tiles_w;
                            tma_load_4d(a_dst, mA, 0, m0, ck, h, &full[s]);
                            if (p.wg_tpt > 0) {
                                const int first = tc.nt * p.wg_tpt;
                                for (int j = 0; j < p.wg_tpt && first + j < 9; ++j) {
                                    const int tp = first + j;
                                    tma_load_4d(b_dst + j * p.wg_rows * 128, mB, 0, 0, ck + (tp % 3 - p.pad) * p.wg_cshift,
                                                h + tp / 3 - p.pad, &full[s]);
                                }
                            } else {
                                tma_load_4d(b_dst, mB, 0, n0, ck + (tap % 3 - p.pad) * p.wg_cshift, h + tap / 3 - p.pad,
                                            &full[s]);
                            }
                        } else {  // CONV_WGRAD: dy^T {Wo*N, Ho, Cout}, x^T {W*N, H, Cin}
                            const int h = kt / p.tiles_w;
                            const int c0 = (kt % p.tiles_w) * TC_BK;
                            tma_load_3d(a_dst, mA, c0, h, m0, &full[s]);
                            if (p.wg_tpt > 0) {
                                const int first = tc.nt * p.wg_tpt;
                                for (int j = 0; j < p.wg_tpt && first + j < 9; ++j) {
                                    const int tp = first + j;
                                    tma_load_3d(b_dst + j * p.wg_rows * 128, mB, c0 + (tp % 3 - p.pad) * p.img_n,
                                                h + tp / 3 - p.pad, 0, &full[s]);
                                }
                            } else {
                                tma_load_3d(b_dst, mB, c0 + (tap % 3 - p.pad) * p.img_n, h + tap / 3 - p.pad, n0,
                                            &full[s]);
                            }
                        }
                    }
                }
            }
            // every copy issued above has landed before the CTA (and, for a pair,
            // its peer, which waits at the final cluster barrier) may exit
            if (rank == 0) {
                const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
                for (uint32_t k = first; k < it; ++k)
                    if (!mbar_wait_bounded(&full[k % STAGES], (k / STAGES) & 1, p.status, DEV_FLAG_WAIT_PRODUCER))
                        break;
            }
        }
    } else if (warp == 5) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0 && rank == 0) {
            uint32_t it = 0, j = 0;
            bool alive = true;
            for (int t = unit0; t < p.num_tiles && alive; t += units, ++j) {
                const TileCoord tc = own_coord(t);
                int kt0, nkt, tap;
                k_range(tc, kt0, nkt, tap);
                const uint32_t b = j & 1, tph = (j >> 1) & 1;
                if (!mbar_wait_bounded(&tmem_empty[b], tph ^ 1, p.status, DEV_FLAG_WAIT_MMA)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * ACC_STRIDE;
                for (int i = 0; i < nkt; i += KS, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait_bounded(&full[s], ph, p.status, DEV_FLAG_WAIT_MMA)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    const int nq = nkt - i < KS ? nkt - i : KS;
                    for (int q = 0; q < nq; ++q) {
                        const uint32_t a_base = smem_u32(sA + (s * KS + q) * TC_A_STAGE);
                        const uint32_t b_base = smem_u32(sB + (s * KS + q) * B_STAGE);
#pragma unroll
                        for (int kk = 0; kk < TC_BK / 8; ++kk) {
                            // K-major, 128-byte swizzle: 8 rows of 128 B per 1024-byte group (SBO);
                            // each K=8 step advances 32 bytes inside the swizzled row.
                            const uint64_t da = smem_desc_sw128(a_base + kk * 32, 16, 1024);
                            const uint64_t db = smem_desc_sw128(b_base + kk * 32, 16, 1024);
                            const uint32_t acc = (i > 0 || q > 0 || kk > 0) ? 1u : 0u;
                            if constexpr (PAIR)
                                mma_tf32_pair(d_tmem, da, db, IDESC, acc);
                            else
                                mma_tf32(d_tmem, da, db, IDESC, acc);
                        }
                    }
                    if constexpr (PAIR)
                        mma_commit_pair(&empty[s], 0x3);
                    else
                        mma_commit(&empty[s]);
                }
                if constexpr (PAIR)
                    mma_commit_pair(&tmem_full[b], 0x3);
                else
                    mma_commit(&tmem_full[b]);
            }
            // every MMA issued above has completed once this commit arrives
            if constexpr (PAIR)
                mma_commit_pair(mma_done, 0x1);
            else
                mma_commit(mma_done);
            mbar_wait_bounded(mma_done, 0, p.status, DEV_FLAG_WAIT_MMA);
        }
        __syncwarp();
    } else if (ROLE == ROLE_CONV_RGB && warp >= 6) {
        // ---------------------------------------------------------------- CONV_RGB im2col rows (warps 6-9)
        // lane l of warp 6 + i writes tile row 32 i + l: ((dh * 3 + dw) * 3 + c) -> x at (h + dh - 1,
        // w + dw - 1), zero outside the image and past k = 27, 128B-swizzled as TMA would; the
        // generic-proxy stores are fenced before the warp's arrival on the stage
        uint32_t it = 0;
        const long long npix = p.M;
        const int hw = p.out_h * p.out_w;
        const int r = (warp - 6) * 32 + lane;
        for (int t = unit0; t < p.num_tiles; t += units, ++it) {
            const uint32_t s = it % STAGES;
            if (!mbar_wait_bounded(&empty[s], ((it / STAGES) & 1) ^ 1, p.status, DEV_FLAG_WAIT_PRODUCER)) break;
            const int pix = (t % p.m_tiles) * TC_BM + r;   // < 2^31 (checked by the host)
            float v[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = 0.f;
            if (pix < npix) {
                const int n = pix / hw;
                const int rem = pix - n * hw;
                const int h = rem / p.out_w, w = rem - h * p.out_w;
                const float* xi = p.act + static_cast<long long>(n) * hw * 3;
#pragma unroll
                for (int dh = 0; dh < 3; ++dh) {
                    const int hh = h + dh - 1;
                    if (hh < 0 || hh >= p.out_h) continue;
                    const float* xr = xi + static_cast<long long>(hh) * p.out_w * 3;
#pragma unroll
                    for (int dw = 0; dw < 3; ++dw) {
                        const int ww = w + dw - 1;
                        if (ww < 0 || ww >= p.out_w) continue;
#pragma unroll
                        for (int c = 0; c < 3; ++c) v[(dh * 3 + dw) * 3 + c] = xr[ww * 3 + c];
                    }
                }
            }
            uint8_t* a_dst = sA + s * KS * TC_A_STAGE;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                *reinterpret_cast<float4*>(a_dst + r * 128 + ((k ^ (r & 7)) << 4)) =
                    make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[s]);
        }
    } else {
        // ---------------------------------------------------------------- epilogue (warps 0-3)
        uint8_t* stage = sStage + warp * NSTG * 4096;
        bool pending = false;     // a TMA store of this warp may still read `stage`
        uint32_t nst = 0;         // chunks this warp has staged (buffer nst % NSTG)
        uint32_t j = 0;
        for (int t = unit0; t < p.num_tiles; t += units, ++j) {
            const TileCoord tc = own_coord(t);
            int kt0, nkt, tap;
            k_range(tc, kt0, nkt, tap);
            const uint32_t b = j & 1, tph = (j >> 1) & 1;
            bool ok = mbar_wait_bounded(&tmem_full[b], tph, p.status, DEV_FLAG_WAIT_EPILOGUE);
            if constexpr (ROLE == ROLE_CONV_RGB) {   // the four warps go on together, or none
                uint32_t all;
                asm volatile(
                    "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 2, 128, p;\n\t"
                    "selp.u32 %0, 1, 0, q;\n\t}"
                    : "=r"(all)
                    : "r"(ok ? 1u : 0u)
                    : "memory");
                ok = all != 0;
            }
            if (!ok) break;
            tc_fence_after();
            const int n0 = tc.nt * BN, m0 = tc.mt * TC_BM;
            const CUtensorMap* mD = &maps.d[G > 1 ? tc.z : 0];
            const float* bias = G > 1 ? p.g_bias[tc.z] : p.bias;
            const float* mask = G > 1 ? p.g_mask[tc.z] : p.mask;
            float* Dout = G > 1 ? p.g_D[tc.z] : p.D;
            const int r = warp * 32 + lane;  // tile row = TMEM lane
            if (tc.tail >= 0) {
                // a k-range of a tail tile: park the raw accumulator rows in the slab
                float* slab = p.tail_part +
                              (static_cast<long long>(tc.tail) * (PAIR ? 2 * TC_BM : TC_BM) + rank * TC_BM + r) * BN;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem_base + b * ACC_STRIDE + (static_cast<uint32_t>(warp * 32) << 16) + c, v);
                    tmem_wait_ld();
                    if (c + 32 >= BN) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (PAIR)
                                mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tmem_empty[b]), 0));
                            else
                                mbar_arrive_cluster_relaxed(smem_u32(&tmem_empty[b]));
                        }
                    }
                    if (nkt == 0) {   // an empty k-range contributes zeros (the accumulator was never written)
#pragma unroll
                        for (int q = 0; q < 32; ++q) v[q] = 0u;
                    }
#pragma unroll
                    for (int q = 0; q < 32; q += 4)
                        *reinterpret_cast<float4*>(slab + c + q) =
                            make_float4(__uint_as_float(v[q]), __uint_as_float(v[q + 1]), __uint_as_float(v[q + 2]),
                                        __uint_as_float(v[q + 3]));
                }
                continue;
            }
            if constexpr (ROLE == ROLE_CONV_RGB) {
                // the tile's 128 rows x 64 channels leave as two TMA boxes of 128 rows x 32 channels,
                // written by the four warps into one of two 32 KB buffers (tile parity); warp 0 waits
                // for the buffer's stores of two tiles ago and issues the new ones
                uint8_t* buf = sStage + (j & 1) * 32768;
                if (warp == 0 && lane == 0 && j >= 2) bulk_wait_read<1>();
                asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll 1
                for (int c = 0; c < 64; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem_base + b * ACC_STRIDE + (static_cast<uint32_t>(warp * 32) << 16) + c, v);
                    tmem_wait_ld();
                    if (c == 32) {   // accumulator fully read: hand it back to the MMA warp
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster_relaxed(smem_u32(&tmem_empty[b]));
                    }
                    float o[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        float x = __uint_as_float(v[q]);
                        if (bias) x += bias[c + q];
                        o[q] = p.relu ? fmaxf(x, 0.f) : x;
                    }
                    uint8_t* half = buf + (c / 32) * 16384;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<float4*>(half + r * 128 + ((q ^ (r & 7)) << 4)) =
                            make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                }
                fence_async_smem();
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (warp == 0 && lane == 0) {
                    tma_store_2d(mD, 0, m0, buf);
                    tma_store_2d(mD, 32, m0, buf + 16384);
                    bulk_commit();
                }
                continue;
            }
            if constexpr (ROLE == ROLE_CONV_FACT) {
                // lane l of warp k is pixel w0 + 30k - 1 + l of the tile's image row; lanes 1-30
                // output the sum of block dw1 of their own row and blocks dw0 / dw2 of rows l - s
                // and l + s of the same window (shuffles), then go out as one 30-pixel TMA box
                int fn, fh, fw0;
                fact_tile(p, tc.mt, fn, fh, fw0);
                const int wfirst = fw0 + warp * TC_FACT_WIN;   // the window's first output pixel
                const int w = wfirst - 1 + lane;
                const bool out_row = fn < p.img_n && lane >= 1 && lane <= TC_FACT_WIN && w < p.out_w;
                const long long pix = (static_cast<long long>(fn) * p.out_h + fh) * p.out_w + w;
                const int lo_blk = p.tap_sign > 0 ? 0 : 2;   // block taken from row l - 1
                const int hi_blk = 2 - lo_blk;                // block taken from row l + 1
                const bool box_inside = fn < p.img_n && wfirst < p.out_w;
#pragma unroll 1
                for (int jb = 0; jb < 2; ++jb) {   // the two 32-channel halves of the 64 outputs
                    uint32_t vl[32], vm[32], vh[32];
                    const uint32_t tb = tmem_base + b * ACC_STRIDE + (static_cast<uint32_t>(warp * 32) << 16);
                    tmem_ld_32x32b_x32(tb + lo_blk * 64 + jb * 32, vl);
                    tmem_ld_32x32b_x32(tb + 64 + jb * 32, vm);
                    tmem_ld_32x32b_x32(tb + hi_blk * 64 + jb * 32, vh);
                    tmem_wait_ld();
                    if (jb == 1) {   // accumulator fully read: hand it back to the MMA warp
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tmem_empty[b]), 0));
                    }
                    const int c0 = jb * 32;
                    float o[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q)
                        o[q] = __shfl_up_sync(0xffffffffu, __uint_as_float(vl[q]), 1) + __uint_as_float(vm[q]) +
                               __shfl_down_sync(0xffffffffu, __uint_as_float(vh[q]), 1);
                    if (p.epi == EPI_STORE) {
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            const float x = o[q] + (p.bias ? p.bias[c0 + q] : 0.f);
                            o[q] = p.relu ? fmaxf(x, 0.f) : x;
                        }
                    } else if (p.mask) {
                        // EPI_MASK: the ReLU mask of the layer below. The window's 32 pixel rows x 32
                        // channels are read row-contiguously by the warp (8 lanes per 128-byte row) into
                        // the staging rows, then each lane takes its own row
                        if (pending) {
                            if (lane == 0) bulk_wait_read0();
                            __syncwarp();
                            pending = false;
                        }
#pragma unroll
                        for (int it = 0; it < 8; ++it) {
                            const int row = it * 4 + (lane >> 3), cq = lane & 7;
                            const int wr = wfirst - 1 + row;
                            float4 mv = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (fn < p.img_n && wr >= 0 && wr < p.out_w)
                                mv = *reinterpret_cast<const float4*>(
                                    p.mask + ((static_cast<long long>(fn) * p.out_h + fh) * p.out_w + wr) * p.ldm + c0 +
                                    4 * cq);
                            *reinterpret_cast<float4*>(stage + row * 128 + ((cq ^ (row & 7)) << 4)) = mv;
                        }
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 mv = *reinterpret_cast<const float4*>(stage + lane * 128 + ((q ^ (lane & 7)) << 4));
                            o[4 * q] = mv.x > 0.f ? o[4 * q] : 0.f;
                            o[4 * q + 1] = mv.y > 0.f ? o[4 * q + 1] : 0.f;
                            o[4 * q + 2] = mv.z > 0.f ? o[4 * q + 2] : 0.f;
                            o[4 * q + 3] = mv.w > 0.f ? o[4 * q + 3] : 0.f;
                        }
                        __syncwarp();   // the output staging below rewrites these rows
                    }
                    if (p.store == ST_PIX4D) {
                        // rows 1-30 staged as smem rows 0-29 (128B-swizzled), one TMA box of 30 pixels;
                        // TMA clips the pixels past the image
                        if (pending) {
                            if (lane == 0) bulk_wait_read0();
                            __syncwarp();
                        }
                        if (lane >= 1 && lane <= TC_FACT_WIN) {
                            const int sr = lane - 1;
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                *reinterpret_cast<float4*>(stage + sr * 128 + ((q ^ (sr & 7)) << 4)) =
                                    make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                        }
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0 && box_inside) {
                            tma_store_4d(mD, c0, wfirst, fh, fn, stage);
                            bulk_commit();
                        }
                        pending = true;
                    } else if (out_row) {
                        float* dst = p.D + pix * p.ldd + c0;
#pragma unroll
                        for (int q = 0; q < 32; q += 4)
                            *reinterpret_cast<float4*>(dst + q) = make_float4(o[q], o[q + 1], o[q + 2], o[q + 3]);
                    }
                }
                continue;
            }
            if constexpr (ROLE == ROLE_CONV_WGRAD && PAIR && BN == 192) {
                if (p.wg_fact) {
                    // factored weight gradient (Cin = Cout = 64): row r is (dh, ci) = (r / 64, r % 64) in the
                    // even CTA and (2, r) for r < 64 in the odd one; column c is (dw, co) = (c / 64, c % 64)
                    float* slab = p.partial + static_cast<long long>(tc.z) * p.wg_slab;
                    const int dh = rank == 0 ? r / 64 : 2, ci = r % 64;
                    const bool w_row = rank == 0 || r < 64;
#pragma unroll 1
                    for (int c = 0; c < BN; c += 32) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(tmem_base + b * ACC_STRIDE + (static_cast<uint32_t>(warp * 32) << 16) + c,
                                           v);
                        tmem_wait_ld();
                        if (c + 32 >= BN) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tmem_empty[b]), 0));
                        }
                        if (nkt == 0) {
#pragma unroll
                            for (int q = 0; q < 32; ++q) v[q] = 0u;
                        }
                        const int dw = c / 64, co0 = c % 64;
                        if (w_row) {
                            // dW[co][dh * 3 + dw][ci]: lanes hold consecutive ci, one 128-byte store per column
                            float* dst = slab + (static_cast<long long>(co0) * 9 + dh * 3 + dw) * 64 + ci;
#pragma unroll
                            for (int q = 0; q < 32; ++q) dst[q * 9 * 64] = __uint_as_float(v[q]);
                        }
                    }
                    continue;
                }
            }
            // output row of this thread (direct stores, mask loads); -1 if outside
            long long row_off = -1, mask_off = -1;
            int pw0 = 0, ph0 = 0, pn0 = 0;
            if constexpr (ROLE == ROLE_CONV_IMPL) {
                pw0 = (tc.mt % p.tiles_w) * p.bw;
                ph0 = ((tc.mt / p.tiles_w) % p.tiles_h) * p.bh;
                pn0 = (tc.mt / (p.tiles_w * p.tiles_h)) * p.bimg;
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
                }
            }
            const bool to_partial = p.partial != nullptr;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem_base + b * ACC_STRIDE + (static_cast<uint32_t>(warp * 32) << 16) + c, v);
                tmem_wait_ld();
                if (c + 32 >= BN) {  // accumulator fully read: hand it back to the MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR)
                            mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tmem_empty[b]), 0));
                        else
                            mbar_arrive_cluster_relaxed(smem_u32(&tmem_empty[b]));
                    }
                }
                const int ncol0 = n0 + c;
                if (ncol0 >= p.N) continue;  // whole chunk outside the output (warp-uniform)
                float o[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) o[q] = __uint_as_float(v[q]);
                if (!to_partial) {
                    if (p.epi == EPI_STORE) {
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            float x = o[q];
                            if (bias && ncol0 + q < p.N) x += bias[ncol0 + q];
                            if (p.relu) x = fmaxf(x, 0.f);
                            o[q] = x;
                        }
                    } else if (p.epi == EPI_MASK) {
                        if (mask && mask_off >= 0) {
                            const float* ms = mask + mask_off + ncol0;
                            if (ncol0 + 32 <= p.N && (p.ldm & 3) == 0) {
#pragma unroll
                                for (int q = 0; q < 32; q += 4) {
                                    const float4 mv = *reinterpret_cast<const float4*>(ms + q);
                                    o[q] = mv.x > 0.f ? o[q] : 0.f;
                                    o[q + 1] = mv.y > 0.f ? o[q + 1] : 0.f;
                                    o[q + 2] = mv.z > 0.f ? o[q + 2] : 0.f;
                                    o[q + 3] = mv.w > 0.f ? o[q + 3] : 0.f;
                                }
                            } else {
#pragma unroll
                                for (int q = 0; q < 32; ++q)
                                    if (ncol0 + q < p.N) o[q] = ms[q] > 0.f ? o[q] : 0.f;
                            }
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 32; ++q) o[q] *= p.alpha;
                    }
                }
                // columns of D (the vector column, if any, is stored apart)
                const int ncols = (G > 1 && p.vec_col >= 0) ? p.vec_col : p.N;
                if constexpr (G > 1) {
                    if (!to_partial && row_off >= 0) {
                        const long long m = m0 + r;
                        if (p.vec_col >= ncol0 && p.vec_col < ncol0 + 32) {
                            float x = 0.f;
#pragma unroll
                            for (int q = 0; q < 32; ++q)
                                if (ncol0 + q == p.vec_col) x = o[q];
                            float* vp = p.g_vec[tc.z] + m;
                            if (p.accumulate) x += *vp;
                            *vp = x;
                        }
                        float* DT = p.g_DT[tc.z];
                        if (DT) {
                            // lanes hold consecutive rows: each column is one 128-byte warp store
                            DT += static_cast<long long>(ncol0) * p.lddT + m;
#pragma unroll
                            for (int q = 0; q < 32; ++q)
                                if (ncol0 + q < ncols) DT[q * p.lddT] = o[q];
                        }
                    }
                }
                if (p.store != ST_DIRECT) {
                    // stage the 32 x 32 chunk (128B-swizzled rows) and hand it to TMA; the buffer's
                    // previous store (NSTG chunks ago) must have read it
                    uint8_t* sbuf = stage + (nst % NSTG) * 4096;
                    if (nst >= static_cast<uint32_t>(NSTG)) {
                        if (lane == 0) bulk_wait_read<NSTG - 1>();
                        __syncwarp();
                    }
                    ++nst;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float4* dst = reinterpret_cast<float4*>(sbuf + lane * 128 + ((q ^ (lane & 7)) << 4));
                        *dst = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                    }
                    fence_async_smem();
                    __syncwarp();
                    // a box whose origin lies past the output (all 32 rows outside) is not issued
                    bool inside;
                    if constexpr (ROLE == ROLE_CONV_IMPL) {
                        const int row0 = warp * 32;
                        inside = pw0 + row0 % p.bw < p.out_w && ph0 + (row0 / p.bw) % p.bh < p.out_h &&
                                 pn0 + row0 / (p.bw * p.bh) < p.img_n;
                    } else {
                        inside = m0 + warp * 32 < p.M && ncol0 < ncols;
                    }
                    if (lane == 0 && inside) {
                        const bool add = (p.epi == EPI_ACCUM) && p.accumulate && !to_partial;
                        if (p.store == ST_2D) {
                            if (add)
                                tma_reduce_add_2d(mD, ncol0, m0 + warp * 32, sbuf);
                            else
                                tma_store_2d(mD, ncol0, m0 + warp * 32, sbuf);
                        } else if (p.store == ST_PIX4D) {
                            const int row0 = warp * 32;
                            const int wo = row0 % p.bw, ho = (row0 / p.bw) % p.bh, no = row0 / (p.bw * p.bh);
                            tma_store_4d(mD, ncol0, pw0 + wo, ph0 + ho, pn0 + no, sbuf);
                        } else if (p.store == ST_WGRAD3D) {
                            if (add)
                                tma_reduce_add_3d(mD, ncol0, tap, m0 + warp * 32, sbuf);
                            else
                                tma_store_3d(mD, ncol0, tap, m0 + warp * 32, sbuf);
                        } else {  // ST_PARTIAL3D
                            tma_store_3d(mD, ncol0, m0 + warp * 32, tc.z, sbuf);
                        }
                        bulk_commit();
                    }
                    continue;
                }
                // direct stores (outputs TMA cannot describe)
                if (row_off < 0) continue;
                if (to_partial) {
                    float* dst = p.partial + (static_cast<long long>(tc.z) * p.M + (m0 + r)) * p.N + ncol0;
#pragma unroll
                    for (int q = 0; q < 32; ++q)
                        if (ncol0 + q < p.N) dst[q] = o[q];
                    continue;
                }
                long long col_shift = 0;
                if constexpr (ROLE == ROLE_CONV_WGRAD) col_shift = static_cast<long long>(tap) * p.N;
                float* dst = Dout + row_off + col_shift + ncol0;
                const bool vec = (ncol0 + 32 <= ncols) && (p.ldd & 3) == 0;
                if (p.epi == EPI_ACCUM && p.accumulate) {
#pragma unroll
                    for (int q = 0; q < 32; ++q)
                        if (ncol0 + q < ncols) o[q] += dst[q];
                }
                if (vec) {
#pragma unroll
                    for (int q = 0; q < 32; q += 4)
                        *reinterpret_cast<float4*>(dst + q) = make_float4(o[q], o[q + 1], o[q + 2], o[q + 3]);
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q)
                        if (ncol0 + q < ncols) dst[q] = o[q];
                }
            }
        }
        if (lane == 0) bulk_wait0();   // every TMA store of this warp has completed
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();   // neither CTA leaves while the other may still signal it
    if (warp == 5) {
        tc_fence_after();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// Finishes the tail-split tiles of a GEMM_2D launch: out = epilogue(sum of
// the tile's tail_splits slabs, added in k-range order). A block takes one
// 32 x 32 patch of a tile at a time, a thread 4 consecutive columns of one
// patch row (8 threads cover a 128-byte row segment); the transposed copy, if
// any, goes out through shared memory so that its stores are row segments too.
// TM = 256 (pair) or 128.
template <int BN, int TM, int ROLE>
__global__ void __launch_bounds__(256) tc_tail_reduce(const TcParams p, int tail_tiles) {
    __shared__ float patch[32][33];
    if (p.m_tiles <= 0 || p.n_tiles <= 0) return;
    constexpr int PR = TM / 32, PC = BN / 32;   // patches per tile: rows, columns
    const long long patches = static_cast<long long>(tail_tiles) * PR * PC;
    const int prow = threadIdx.x >> 3, pcol = (threadIdx.x & 7) * 4;
    const bool grouped = p.z_tiles > 1 || p.g_D[0] != nullptr;
    for (long long pi = blockIdx.x; pi < patches; pi += gridDim.x) {
        const int j = static_cast<int>(pi / (PR * PC));
        const int rem = static_cast<int>(pi % (PR * PC));
        const int row0 = (rem / PC) * 32, col0 = (rem % PC) * 32;
        // decompose the tile as the kernel did (units are m-fastest; a pair unit spans TM rows)
        const int tt = p.tail_start + j;
        const int mu = tt % p.m_tiles, rr = tt / p.m_tiles;
        const int nt = p.z_mid ? rr / p.z_tiles : rr % p.n_tiles;
        const int z = p.z_mid ? rr % p.z_tiles : rr / p.n_tiles;
        if (z >= p.z_tiles || z >= TC_MAX_GROUP || nt * BN + col0 >= p.N) continue;   // whole patch (uniform)
        const int row = row0 + prow, col = col0 + pcol;
        const int n0 = nt * BN + col;
        long long m = -1;   // output row (GEMM_2D) or output pixel (CONV_IMPL) of this slab row; -1 outside
        if constexpr (ROLE == ROLE_CONV_IMPL) {
            // slab row = rank * 128 + r of the unit's box(es); the box decomposition of the epilogue
            const int mt = TM == 256 ? 2 * mu + row / 128 : mu, r = row % 128;
            const int ow = (mt % p.tiles_w) * p.bw + r % p.bw;
            const int oh = ((mt / p.tiles_w) % p.tiles_h) * p.bh + (r / p.bw) % p.bh;
            const int on = (mt / (p.tiles_w * p.tiles_h)) * p.bimg + r / (p.bw * p.bh);
            if (ow < p.out_w && oh < p.out_h && on < p.img_n)
                m = (static_cast<long long>(on) * p.out_h + oh) * p.out_w + ow;
        } else {
            m = static_cast<long long>(mu) * TM + row;
            if (m >= p.M) m = -1;
        }
        float* D = grouped ? p.g_D[z] : p.D;
        const float* bias = grouped ? p.g_bias[z] : p.bias;
        const float* mask = grouped ? p.g_mask[z] : p.mask;
        float* DT = (ROLE == ROLE_GEMM_2D && grouped) ? p.g_DT[z] : nullptr;
        float* vec = (ROLE == ROLE_GEMM_2D && grouped && p.vec_col >= 0) ? p.g_vec[z] : nullptr;
        const int ncols = vec ? p.vec_col : p.N;
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        if (m >= 0 && n0 < p.N) {
            // the slabs in k-range order; eight loads in flight before their adds (same order)
            const float* slab0 = p.tail_part + (static_cast<long long>(j) * p.tail_splits * TM + row) * BN + col;
            const long long slab_step = static_cast<long long>(TM) * BN;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            int sp = 0;
            for (; sp + 8 <= p.tail_splits; sp += 8) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = *reinterpret_cast<const float4*>(slab0 + (sp + u) * slab_step);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    acc.x += v[u].x;
                    acc.y += v[u].y;
                    acc.z += v[u].z;
                    acc.w += v[u].w;
                }
            }
            for (; sp < p.tail_splits; ++sp) {
                const float4 v = *reinterpret_cast<const float4*>(slab0 + sp * slab_step);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            o[0] = acc.x;
            o[1] = acc.y;
            o[2] = acc.z;
            o[3] = acc.w;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = n0 + q;
                if (n >= p.N || n > ncols) break;
                float x = o[q];
                float* d = (n < ncols) ? D + m * p.ldd + n : vec + m;
                if (p.epi == EPI_STORE) {
                    if (bias) x += bias[n];
                    if (p.relu) x = fmaxf(x, 0.f);
                } else if (p.epi == EPI_MASK) {
                    if (mask && !(mask[m * p.ldm + n] > 0.f)) x = 0.f;
                } else {
                    x *= p.alpha;
                    if (p.accumulate) x += *d;
                }
                o[q] = x;
                *d = x;
            }
        }
        if (DT) {   // uniform over the block
#pragma unroll
            for (int q = 0; q < 4; ++q) patch[prow][pcol + q] = o[q];
            __syncthreads();
            const int c = threadIdx.x >> 3, r0 = (threadIdx.x & 7) * 4;   // patch column, first of 4 rows
            const int n = nt * BN + col0 + c;
            const long long mb = static_cast<long long>(mu) * TM + row0 + r0;
            if (n < ncols) {
                float* dt = DT + static_cast<long long>(n) * p.lddT + mb;
                if (mb + 4 <= p.M && (p.lddT & 3) == 0 && (mb & 3) == 0) {
                    *reinterpret_cast<float4*>(dt) =
                        make_float4(patch[r0][c], patch[r0 + 1][c], patch[r0 + 2][c], patch[r0 + 3][c]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (mb + q < p.M) dt[q] = patch[r0 + q][c];
                }
            }
            __syncthreads();
        }
    }
}

#endif  // __CUDACC__

}  // namespace sprint
