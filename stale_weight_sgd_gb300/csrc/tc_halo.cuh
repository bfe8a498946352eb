// Halo-staged implicit-GEMM 3x3 convolution (pad 1) on tcgen05 CTA pairs: the
// forward pass (y = relu(x * w + b), SPRINT report Sec. 3.3 "convolution")
// and the input gradient (dx = (dy * w^T) . [x > 0], "dedx conv") of layers
// with 64 or 128 output channels.
//
// A CTA's tile is bh output rows x bw output pixels of one image. Its operand
// A comes from a halo buffer: the (bh + 2) x pitch input pixels around the
// tile (pitch = bw + 2), one 32-channel chunk (128 bytes) per pixel row,
// loaded by one TMA box per chunk (zero fill outside the image) and 128-byte
// swizzled. The MMA's 128 rows are the tile positions q = r * pitch + c
// (r < bh, c < pitch): output (r, c) needs buffer row q + dh * pitch + dw for
// the tap (dh, dw) of the forward pass, so a tap's A operand is the 128-row
// window of the buffer that starts dh * pitch + dw rows in. The swizzle is a
// function of the shared-memory address, so an operand may start on any
// 128-byte row (measured: exact products for row offsets 1-31). One chunk
// thus reads ~(bh + 2) * pitch pixel rows instead of nine 128-row boxes.
// Positions with c >= bw (the two columns the pitch adds) are not stored.
//
// Two forms, by the width of one MMA (a CTA-pair MMA with N <= 128 takes ~123
// cycles however narrow it is, so narrow tiles waste the tensor core):
//  - BN = 128 (128 output channels): per chunk, the nine taps' windows against
//    the tap's weight slice (B stages of one kernel row, three taps each);
//    the input gradient takes the mirrored tap's window, (2 - dh) * pitch +
//    (2 - dw).
//  - BN = 192 (64 output channels), factored over the kernel columns: B' =
//    the weights permuted to rows (dw, c) and columns (dh, k), so that per
//    chunk three windows (dh * pitch rows in; (2 - dh) * pitch for the input
//    gradient) give D'[q][(dw, c)] = sum over dh, k of A[q + dh * pitch][k] *
//    w[c][dh][dw][k], and the epilogue adds out[q] = D'[q][0] + D'[q + 1][1] +
//    D'[q + 2][2] (input gradient: D'[q + 2][0] + D'[q + 1][1] + D'[q][2]):
//    rows q + 1 and q + 2 come from the next lanes of the warp, and for a
//    warp's last two lanes from the next warp through shared memory. The
//    largest row a stored output needs is bh * pitch - 1 < 128, inside the
//    tile.
//
// Warp roles: warp 8 lane 0 loads (both CTAs, each its own halo buffer and
// half of the B rows, completing on the even CTA's barriers); warp 9 lane 0 of
// the even CTA issues the M = 256 MMAs; warps 0-7 drain the accumulator
// (double-buffered in TMEM; warps w and w + 4 read the same 32 TMEM lanes and
// take alternate 32-column chunks, two warps per sub-partition to hide the
// epilogue's latencies) and store through a small staging area as whole
// 128-byte rows (a warp's 32 positions can span two output rows). Two rings: the
// halo buffers (one per chunk) and the B stages (three k-tiles each). Every
// wait is bounded; one that gives up sets a bit of the device status word and
// the CTA finishes. An epilogue warp hands its part of the accumulator back with
// a relaxed arrive: a release would first wait for the warp's earlier output
// stores to become visible (the epilogue warps agree on giving up through a barrier
// reduction, so none is left at a named barrier).
#pragma once

#include "tc_gemm.cuh"

namespace sprint {

constexpr int HALO_A_BYTES = 45 * 1024;              // one halo buffer: at most 360 pixel rows of 128 B
constexpr int HALO_A_ROWS = HALO_A_BYTES / 128;

// rows of the buffer the MMAs read: the last tap's window ends 2 * pitch + 2 + 128 rows in
__host__ __device__ constexpr int halo_rows_needed(int bw, int bh) {
    return ((bh + 2) * (bw + 2) > 2 * (bw + 2) + 2 + TC_BM ? (bh + 2) * (bw + 2) : 2 * (bw + 2) + 2 + TC_BM);
}
// ring depths: halo buffers, and B stages of three k-tiles (a pair's half of the BN rows each)
__host__ __device__ constexpr int halo_a_stages(int bn) { return bn == 192 ? 2 : (bn >= 128 ? 2 : 3); }
__host__ __device__ constexpr int halo_b_stage(int bn) { return 3 * (bn / 2) * TC_BK * 4; }
__host__ __device__ constexpr int halo_b_stages(int bn) { return bn == 192 ? 2 : (bn >= 128 ? 5 : 6); }
// BN = 192: the edge rows the epilogue warps pass on (two co halves x 4 warps x 3 rows x 32 floats)
constexpr int HALO_XCH_BYTES = 2 * 4 * 3 * 32 * 4;
// warps 0-7 drain the accumulator (warps w and w + 4 share TMEM lanes 32 (w % 4) .. + 31 and split
// its columns), warp 8 loads, warp 9 issues the MMAs
constexpr int HALO_THREADS = 320;
// per epilogue warp: rows of 128 B through which its stores (and mask loads) go out as whole rows;
// BN = 192 has a 32-row (4 KB) box per warp for its TMA mask loads and stores
__host__ __device__ constexpr int halo_stg_warp(int bn) { return bn == 192 ? 32 * 128 : 8 * 128; }
__host__ __device__ constexpr int halo_smem_bytes(int bn) {
    return 1024 + halo_a_stages(bn) * HALO_A_BYTES + halo_b_stages(bn) * halo_b_stage(bn) + 1024 +
           8 * halo_stg_warp(bn) + (bn == 192 ? HALO_XCH_BYTES : 0);
}

// Tensor maps of a halo launch: A (input, halo boxes), B (weights); BN = 192 with halo_tma: D and the
// ReLU mask in boxes of 32 pixels (d, m) and of the row's last bw % 32 (dt, mt), 32 channels each.
struct HaloMaps {
    CUtensorMap a, b, d, dt, m, mt;
};

// CTA tile mt of a halo launch: image n, first output row h0 and pixel w0 (n >= img_n past the
// last tile)
__host__ __device__ __forceinline__ void halo_tile(const TcParams& p, int mt, int& n, int& h0, int& w0) {
    w0 = (mt % p.tiles_w) * p.bw;
    h0 = ((mt / p.tiles_w) % p.tiles_h) * p.bh;
    n = mt / (p.tiles_w * p.tiles_h);
}

#if defined(__CUDACC__)

// The four epilogue warps of column group g (warps 4g .. 4g + 3): named barrier 1 + g, and an AND
// over them (barrier 3 + g).
__device__ __forceinline__ void epi_bar(int g) { asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory"); }
__device__ __forceinline__ bool epi_all(int g, bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(ok ? 1u : 0u), "r"(3 + g)
        : "memory");
    return r != 0;
}

// Row r (0-7) of an epilogue warp's staging area, 16-byte chunk k, 128-byte swizzled.
__device__ __forceinline__ float4* halo_stg(uint8_t* stg, int r, int k) {
    return reinterpret_cast<float4*>(stg + r * 128 + ((k ^ (r & 7)) << 4));
}

// o[] = 32 consecutive columns of lane l's tile row; off = that row's element offset in D (-1: not
// stored). Out through the staging rows, 8 lanes at a time, so that each warp store writes four
// whole 128-byte rows.
__device__ __forceinline__ void halo_store_rows(const float (&o)[32], long long off, float* D, uint8_t* stg, int lane) {
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
        if ((lane >> 3) == pass) {
            const int r = lane & 7;
#pragma unroll
            for (int k = 0; k < 8; ++k) *halo_stg(stg, r, k) = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int rr = 4 * i + (lane >> 3), k = lane & 7;
            const long long so = __shfl_sync(0xffffffffu, off, 8 * pass + rr);
            const float4 v = *halo_stg(stg, rr, k);
            if (so >= 0) *reinterpret_cast<float4*>(D + so + 4 * k) = v;
        }
        __syncwarp();
    }
}

// o[q] = 0 where the mask row's column q is <= 0 (moff: the row's offset in the mask, -1: none);
// the mask comes in as whole 128-byte rows through the staging area.
__device__ __forceinline__ void halo_mask_rows(float (&o)[32], long long moff, const float* mask, uint8_t* stg,
                                               int lane) {
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int rr = 4 * i + (lane >> 3), k = lane & 7;
            const long long mo = __shfl_sync(0xffffffffu, moff, 8 * pass + rr);
            float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
            if (mo >= 0) m = *reinterpret_cast<const float4*>(mask + mo + 4 * k);
            *halo_stg(stg, rr, k) = m;
        }
        __syncwarp();
        if ((lane >> 3) == pass) {
            const int r = lane & 7;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 m = *halo_stg(stg, r, k);
                o[4 * k] = m.x > 0.f ? o[4 * k] : 0.f;
                o[4 * k + 1] = m.y > 0.f ? o[4 * k + 1] : 0.f;
                o[4 * k + 2] = m.z > 0.f ? o[4 * k + 2] : 0.f;
                o[4 * k + 3] = m.w > 0.f ? o[4 * k + 3] : 0.f;
            }
        }
        __syncwarp();
    }
}

// Work units: u = t % m_tiles (a pair of CTA tiles 2u, 2u + 1), n-tile t / m_tiles.
// p: img_n, out_h, out_w (= the input's H, W), bw, bh, tiles_w, tiles_h, chunks (32-channel
// chunks of the reduction), tap_sign (+1 forward, -1 input gradient), b_tap_outer (BN = 128:
// B map coordinates (k, n, tap) if 1, (k, tap, n) if 0; BN = 192: a 2-D map of B' with
// coordinates (k, n), k = dh * 32 * chunks + channel), epi (EPI_STORE: + bias, ReLU if relu;
// EPI_MASK: x 0 where mask <= 0), D / ldd, bias, mask / ldm, N (output channels), status.
template <int BN>
__global__ void __launch_bounds__(HALO_THREADS, 1)
    tc_halo_kernel(const __grid_constant__ HaloMaps maps, const TcParams p) {
    constexpr bool FACT = BN == 192;             // factored over the kernel columns (64 output channels)
    constexpr int SA = halo_a_stages(BN);
    constexpr int SB = halo_b_stages(BN);
    constexpr int GROUPS = FACT ? 1 : 3;         // B stages per chunk (three k-tiles each)
    constexpr int B_STAGE = halo_b_stage(BN);
    constexpr int B_ROWS = BN / 2;
    constexpr int B_KT = B_ROWS * TC_BK * 4;     // one k-tile within a B stage
    constexpr uint32_t IDESC = idesc_tf32(BN, false, false, 256);
    constexpr uint32_t TMEM_COLS = tc_tmem_cols(BN);
    constexpr uint32_t ACC_STRIDE = TMEM_COLS / 2;
    static_assert(BN == 64 || BN == 128 || BN == 192, "halo tiles are 64, 128 or 3 x 64 columns wide");
    static_assert(halo_smem_bytes(BN) <= 232448, "shared memory budget exceeded");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* sA = smem;
    uint8_t* sB = smem + SA * HALO_A_BYTES;
    uint64_t* a_full = reinterpret_cast<uint64_t*>(sB + SB * B_STAGE);   // barriers: 1024 bytes
    uint64_t* a_empty = a_full + SA;
    uint64_t* b_full = a_empty + SA;
    uint64_t* b_empty = b_full + SB;
    uint64_t* tmem_full = b_empty + SB;    // [2]
    uint64_t* tmem_empty = tmem_full + 2;  // [2]
    uint64_t* mma_done = tmem_empty + 2;
    uint64_t* mask_bar = mma_done + 1;     // [8]: an epilogue warp's TMA mask box
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mask_bar + 8);
    uint8_t* sStg = smem + SA * HALO_A_BYTES + SB * B_STAGE + 1024;   // 1024-aligned (128B-swizzled TMA boxes)
    float* xch = reinterpret_cast<float*>(sStg + 8 * halo_stg_warp(BN));                          // BN = 192

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int unit0 = static_cast<int>(blockIdx.x >> 1);
    const int units = static_cast<int>(gridDim.x >> 1);
    const int pitch = p.bw + 2;
    // bytes of one halo box (TMA counts the zero fill too)
    const uint32_t a_bytes = static_cast<uint32_t>((p.bh + 2) * pitch) * 128u;

    if (warp == 8 && lane == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < SB; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tmem_full[b], 1);
            mbar_init(&tmem_empty[b], 16);   // one arrival per epilogue warp of both CTAs
        }
        mbar_init(mma_done, 1);
        for (int w = 0; w < 8; ++w) mbar_init(&mask_bar[w], 1);
        fence_mbar_init();
        tma_prefetch_desc(&maps.a);
        tma_prefetch_desc(&maps.b);
    }
    if (warp == 9) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // the peer's barriers are initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 8) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t ia = 0, ib = 0;
            bool alive = true;
            const CUtensorMap* mA = &maps.a;
            const CUtensorMap* mB = &maps.b;
            for (int t = unit0; t < p.num_tiles && alive; t += units) {
                const int mt = 2 * (t % p.m_tiles) + static_cast<int>(rank);
                const int n0 = (t / p.m_tiles) * BN + static_cast<int>(rank) * B_ROWS;
                int n, h0, w0;
                halo_tile(p, mt, n, h0, w0);
                for (int c = 0; c < p.chunks && alive; ++c) {
                    const uint32_t sa = ia % SA;
                    if (!mbar_wait_bounded(&a_empty[sa], ((ia / SA) & 1) ^ 1, p.status, DEV_FLAG_WAIT_PRODUCER)) {
                        alive = false;
                        break;
                    }
                    if (rank == 0) mbar_arrive_expect_tx(&a_full[sa], 2u * a_bytes);
                    tma_load_4d_pair(sA + sa * HALO_A_BYTES, mA, c * TC_BK, w0 - 1, h0 - 1, n,
                                     mapa_shared(smem_u32(&a_full[sa]), 0));
                    ++ia;
                    for (int g = 0; g < GROUPS; ++g) {
                        const uint32_t sb = ib % SB;
                        if (!mbar_wait_bounded(&b_empty[sb], ((ib / SB) & 1) ^ 1, p.status, DEV_FLAG_WAIT_PRODUCER)) {
                            alive = false;
                            break;
                        }
                        if (rank == 0) mbar_arrive_expect_tx(&b_full[sb], 2u * B_STAGE);
                        const uint32_t bar = mapa_shared(smem_u32(&b_full[sb]), 0);
#pragma unroll
                        for (int u = 0; u < 3; ++u) {
                            uint8_t* dst = sB + sb * B_STAGE + u * B_KT;
                            if constexpr (FACT)   // B' columns of kernel row u, this chunk
                                tma_load_2d_pair(dst, mB, (u * p.chunks + c) * TC_BK, n0, bar);
                            else if (p.b_tap_outer)
                                tma_load_3d_pair(dst, mB, c * TC_BK, n0, 3 * g + u, bar);
                            else
                                tma_load_3d_pair(dst, mB, c * TC_BK, 3 * g + u, n0, bar);
                        }
                        ++ib;
                    }
                }
            }
            // every copy issued above has landed before the CTA (and its peer, which waits at the
            // final cluster barrier) may exit
            if (rank == 0) {
                for (uint32_t k = ia > static_cast<uint32_t>(SA) ? ia - SA : 0u; k < ia; ++k)
                    if (!mbar_wait_bounded(&a_full[k % SA], (k / SA) & 1, p.status, DEV_FLAG_WAIT_PRODUCER)) break;
                for (uint32_t k = ib > static_cast<uint32_t>(SB) ? ib - SB : 0u; k < ib; ++k)
                    if (!mbar_wait_bounded(&b_full[k % SB], (k / SB) & 1, p.status, DEV_FLAG_WAIT_PRODUCER)) break;
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0 && rank == 0) {
            uint32_t ia = 0, ib = 0, j = 0;
            bool alive = true;
            for (int t = unit0; t < p.num_tiles && alive; t += units, ++j) {
                const uint32_t b = j & 1, tph = (j >> 1) & 1;
                if (!mbar_wait_bounded(&tmem_empty[b], tph ^ 1, p.status, DEV_FLAG_WAIT_MMA)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * ACC_STRIDE;
                for (int c = 0; c < p.chunks && alive; ++c) {
                    const uint32_t sa = ia % SA;
                    if (!mbar_wait_bounded(&a_full[sa], (ia / SA) & 1, p.status, DEV_FLAG_WAIT_MMA)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + sa * HALO_A_BYTES);
                    for (int g = 0; g < GROUPS; ++g) {
                        const uint32_t sb = ib % SB;
                        if (!mbar_wait_bounded(&b_full[sb], (ib / SB) & 1, p.status, DEV_FLAG_WAIT_MMA)) {
                            alive = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int u = 0; u < 3; ++u) {
                            // the window of k-tile u: kernel row dh, and column dw unless factored
                            const int dh = FACT ? u : g, dw = FACT ? 0 : u;
                            const int off = p.tap_sign > 0 ? dh * pitch + dw : (2 - dh) * pitch + (FACT ? 0 : 2 - dw);
                            const uint32_t a_win = a_base + static_cast<uint32_t>(off) * 128u;
                            const uint32_t b_base = smem_u32(sB + sb * B_STAGE + u * B_KT);
#pragma unroll
                            for (int kk = 0; kk < TC_BK / 8; ++kk) {
                                const uint64_t da = smem_desc_sw128(a_win + kk * 32, 16, 1024);
                                const uint64_t db = smem_desc_sw128(b_base + kk * 32, 16, 1024);
                                mma_tf32_pair(d_tmem, da, db, IDESC, (c > 0 || g > 0 || u > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                        mma_commit_pair(&b_empty[sb], 0x3);
                        ++ib;
                    }
                    if (!alive) break;
                    mma_commit_pair(&a_empty[sa], 0x3);
                    ++ia;
                }
                mma_commit_pair(&tmem_full[b], 0x3);
            }
            // every MMA issued above has completed once this commit arrives
            mma_commit_pair(mma_done, 0x1);
            mbar_wait_bounded(mma_done, 0, p.status, DEV_FLAG_WAIT_MMA);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue (warps 0-7)
        const int quarter = warp & 3, grp = warp >> 2;   // TMEM lanes 32 * quarter .., column group
        const int r = quarter * 32 + lane;               // tile position = TMEM lane
        const int hr = r / pitch, wc = r % pitch;
        uint8_t* stg = sStg + warp * halo_stg_warp(BN);
        // TMA epilogue (BN = 192, one-row tiles): this warp's pixels w0 + 32 quarter .. (cnt of them)
        const int cnt = p.bw - 32 * quarter < 32 ? p.bw - 32 * quarter : 32;
        const CUtensorMap* mapd = cnt == 32 ? &maps.d : &maps.dt;
        const CUtensorMap* mapm = cnt == 32 ? &maps.m : &maps.mt;
        uint32_t nmask = 0, nmask_issued = 0;   // mask boxes waited for (the barrier's phase) / issued
        bool mask_ok = true;                     // no mask wait has run out
        uint32_t j = 0;
        for (int t = unit0; t < p.num_tiles; t += units, ++j) {
            const int mt = 2 * (t % p.m_tiles) + static_cast<int>(rank);
            const int nt = t / p.m_tiles;
            int n, h0, w0;
            halo_tile(p, mt, n, h0, w0);
            const int oh = h0 + hr, ow = w0 + wc;
            const bool valid = hr < p.bh && wc < p.bw && oh < p.out_h && ow < p.out_w && n < p.img_n;
            const long long pix = (static_cast<long long>(n) * p.out_h + oh) * p.out_w + ow;
            const long long off = valid ? pix * p.ldd : -1;   // this row in D
            const bool masked = p.epi == EPI_MASK && p.mask;
            const long long moff = masked && valid ? pix * p.ldm : -1;
            if (moff >= 0) {   // the mask lines of this warp's chunks on their way to L2 while the MMAs run
#pragma unroll 1
                for (int c = (FACT ? 0 : nt * BN) + 32 * grp; c < (FACT ? 64 : nt * BN + BN) && c < p.N; c += 64)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.mask + moff + c) : "memory");
            }
            // TMA epilogue: the warp's box lies in the image (TMA clips its end at the image edge)
            const bool tbox = FACT && p.halo_tma && cnt > 0 && n < p.img_n && h0 < p.out_h && w0 + 32 * quarter < p.out_w;
            if (tbox && masked) {   // the mask block on its way while the MMAs run
                if (lane == 0) {
                    bulk_wait_read0();   // the buffer's last store has read it
                    mbar_arrive_expect_tx(&mask_bar[warp], static_cast<uint32_t>(cnt) * 128u);
                    tma_load_4d(stg, mapm, 32 * grp, w0 + 32 * quarter, h0, n, &mask_bar[warp]);
                }
                ++nmask_issued;
            }
            const uint32_t b = j & 1, tph = (j >> 1) & 1;
            bool ok = mbar_wait_bounded(&tmem_full[b], tph, p.status, DEV_FLAG_WAIT_EPILOGUE);
            if constexpr (FACT) ok = epi_all(grp, ok && mask_ok);   // the group's four warps go on, or none
            if (!ok) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + b * ACC_STRIDE + (static_cast<uint32_t>(quarter * 32) << 16);
            if constexpr (FACT) {
                const bool fwd = p.tap_sign > 0;
                {   // group g takes 32-channel half jb = g of the 64 outputs
                    const int jb = grp, col = jb * 32;
                    uint32_t v0[32], v1[32], v2[32];   // column blocks dw = 0, 1, 2 of this half
                    __syncwarp();
                    tmem_ld_32x32b_x32(tb + col, v0);
                    tmem_ld_32x32b_x32(tb + 64 + col, v1);
                    tmem_ld_32x32b_x32(tb + 128 + col, v2);
                    tmem_wait_ld();
                    {   // this warp's part of the accumulator is read: hand it back to the MMA warp
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tmem_empty[b]), 0));
                    }
                    // out[q] = a0[q] + v1[q + 1] + a2[q + 2] (a0 / a2 = blocks dw 0 / 2, swapped for the
                    // input gradient); lanes 0 and 1 pass v1 / a2 of their rows on to the previous warp
#define HALO_A0(q) __uint_as_float(fwd ? v0[q] : v2[q])
#define HALO_A2(q) __uint_as_float(fwd ? v2[q] : v0[q])
                    float* xw = xch + (jb * 4 + quarter) * 96;
                    if (lane == 0) {
#pragma unroll
                        for (int q = 0; q < 32; q += 4) {
                            *reinterpret_cast<float4*>(xw + q) =
                                make_float4(__uint_as_float(v1[q]), __uint_as_float(v1[q + 1]),
                                            __uint_as_float(v1[q + 2]), __uint_as_float(v1[q + 3]));
                            *reinterpret_cast<float4*>(xw + 32 + q) =
                                make_float4(HALO_A2(q), HALO_A2(q + 1), HALO_A2(q + 2), HALO_A2(q + 3));
                        }
                    } else if (lane == 1) {
#pragma unroll
                        for (int q = 0; q < 32; q += 4)
                            *reinterpret_cast<float4*>(xw + 64 + q) =
                                make_float4(HALO_A2(q), HALO_A2(q + 1), HALO_A2(q + 2), HALO_A2(q + 3));
                    }
                    float o[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const float s1 = __shfl_down_sync(0xffffffffu, __uint_as_float(v1[q]), 1);
                        const float s2 = __shfl_down_sync(0xffffffffu, HALO_A2(q), 2);
                        o[q] = HALO_A0(q) + (lane < 31 ? s1 : 0.f) + (lane < 30 ? s2 : 0.f);
                    }
#undef HALO_A0
#undef HALO_A2
                    epi_bar(grp);
                    if (lane >= 30 && quarter < 3) {   // the next quarter's first rows (quarter 3 stores no such row)
                        const float* xn = xch + (jb * 4 + quarter + 1) * 96;
#pragma unroll
                        for (int q = 0; q < 32; q += 4) {
                            const float4 t2 = *reinterpret_cast<const float4*>(xn + (lane == 31 ? 64 : 32) + q);
                            const float4 t1 = lane == 31 ? *reinterpret_cast<const float4*>(xn + q)
                                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                            o[q] += t1.x + t2.x;
                            o[q + 1] += t1.y + t2.y;
                            o[q + 2] += t1.z + t2.z;
                            o[q + 3] += t1.w + t2.w;
                        }
                    }
                    if (p.epi == EPI_STORE) {
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            const float x = o[q] + (p.bias ? p.bias[col + q] : 0.f);
                            o[q] = p.relu ? fmaxf(x, 0.f) : x;
                        }
                    } else if (masked && !p.halo_tma) {
                        halo_mask_rows(o, moff >= 0 ? moff + col : -1, p.mask, stg, lane);
                    }
                    if (!p.halo_tma) {
                        halo_store_rows(o, off >= 0 ? off + col : -1, p.D, stg, lane);
                        continue;
                    }
                    if (!tbox) continue;
                    if (masked) {   // lane l's mask row l of the box, 128B-swizzled as TMA wrote it
                        if (!mbar_wait_bounded(&mask_bar[warp], nmask & 1, p.status, DEV_FLAG_WAIT_EPILOGUE))
                            mask_ok = false;   // the group stops at the next tile
                        ++nmask;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float4 m = *reinterpret_cast<const float4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4));
                            o[4 * k] = m.x > 0.f ? o[4 * k] : 0.f;
                            o[4 * k + 1] = m.y > 0.f ? o[4 * k + 1] : 0.f;
                            o[4 * k + 2] = m.z > 0.f ? o[4 * k + 2] : 0.f;
                            o[4 * k + 3] = m.w > 0.f ? o[4 * k + 3] : 0.f;
                        }
                        __syncwarp();   // every lane has read its mask row before the rows are rewritten
                    } else {
                        if (lane == 0) bulk_wait_read0();   // the buffer's last store has read it
                        __syncwarp();
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<float4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                            make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_4d(mapd, col, w0 + 32 * quarter, h0, n, stg);
                        bulk_commit();
                    }
                }
                continue;
            }
#pragma unroll 1
            for (int c = 32 * grp; c < BN; c += 64) {   // group g: 32-column chunks g, g + 2, ...
                const int col = nt * BN + c;
                uint32_t v[32];
                __syncwarp();   // converged for the warp-wide TMEM load
                tmem_ld_32x32b_x32(tb + c, v);
                tmem_wait_ld();
                if (c + 64 >= BN) {   // this warp's part of the accumulator is read: hand it back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tmem_empty[b]), 0));
                }
                if (col >= p.N) continue;   // warp-uniform
                float o[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) o[q] = __uint_as_float(v[q]);
                if (p.epi == EPI_STORE) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const float x = o[q] + (p.bias ? p.bias[col + q] : 0.f);
                        o[q] = p.relu ? fmaxf(x, 0.f) : x;
                    }
                } else if (masked) {
                    halo_mask_rows(o, moff >= 0 ? moff + col : -1, p.mask, stg, lane);
                }
                halo_store_rows(o, off >= 0 ? off + col : -1, p.D, stg, lane);
            }
        }
        // a mask box still in flight (a group that stopped early) lands before the CTA exits
        for (; nmask < nmask_issued; ++nmask) mbar_wait_bounded(&mask_bar[warp], nmask & 1, p.status, DEV_FLAG_WAIT_EPILOGUE);
        if (lane == 0) bulk_wait0();   // every TMA store of this warp has completed
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();   // neither CTA leaves while the other may still signal it
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

#endif  // __CUDACC__

// ---------------------------------------------------------------------------------------------
// 128 output channels with the roles swapped ("flipped"): the weights are the MMA's M = 128
// operand and 256 tile positions its N side, one CTA per tile (M = 128, N = 256: the math rate,
// where the pair tile of N = 128 above sits at the ~123-cycle floor of a narrow MMA). A tile is
// bh output rows of bw pixels with bh * (bw + 2) <= 256 positions; per 32-channel chunk one halo
// box of (bh + 2) x (bw + 2) input pixels, and per tap the B operand is the 256-row window of it
// that starts dh * pitch + dw rows in (the mirrored tap for the input gradient), the A operand the
// tap's 128 x 32 weight slice. The accumulator holds [channel][position]: epilogue warp w reads
// channels 32 (w % 4) .. + 31 (its TMEM lanes) and position chunks w / 4, w / 4 + 2, ..., and
// stores each position's 32 channels as one 128-byte row (bias: one value per lane).
constexpr int HALO_F_POS = 256;                   // tile positions (the MMA's N)
constexpr int HALO_F_A_BYTES = 61 * 1024;         // halo buffer: at most 488 pixel rows
constexpr int HALO_F_SA = 2, HALO_F_SW = 6;       // halo stages; weight stages (one tap each)
constexpr int HALO_F_W_STAGE = TC_BM * TC_BK * 4; // 128 channels x 32 k
constexpr int HALO_F_SMEM = 1024 + HALO_F_SA * HALO_F_A_BYTES + HALO_F_SW * HALO_F_W_STAGE + 1024;
__host__ __device__ constexpr int halo_f_rows_needed(int bw, int bh) {
    return ((bh + 2) * (bw + 2) > 2 * (bw + 2) + 2 + HALO_F_POS ? (bh + 2) * (bw + 2)
                                                                 : 2 * (bw + 2) + 2 + HALO_F_POS);
}

#if defined(__CUDACC__)

// p as for tc_halo_kernel; tiles m_tiles (= num_tiles), N = 128 output channels.
__global__ void __launch_bounds__(HALO_THREADS, 1)
    tc_halo_flip_kernel(const __grid_constant__ HaloMaps maps, const TcParams p) {
    constexpr int SA = HALO_F_SA, SW = HALO_F_SW;
    constexpr uint32_t IDESC = idesc_tf32(HALO_F_POS, false, false, TC_BM);
    constexpr uint32_t TMEM_COLS = 512, ACC_STRIDE = 256;
    static_assert(HALO_F_SMEM <= 232448, "shared memory budget exceeded");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* sH = smem;
    uint8_t* sW = smem + SA * HALO_F_A_BYTES;
    uint64_t* h_full = reinterpret_cast<uint64_t*>(sW + SW * HALO_F_W_STAGE);
    uint64_t* h_empty = h_full + SA;
    uint64_t* w_full = h_empty + SA;
    uint64_t* w_empty = w_full + SW;
    uint64_t* tmem_full = w_empty + SW;     // [2]
    uint64_t* tmem_empty = tmem_full + 2;   // [2]
    uint64_t* mma_done = tmem_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int pitch = p.bw + 2;
    const uint32_t h_bytes = static_cast<uint32_t>((p.bh + 2) * pitch) * 128u;

    if (warp == 8 && lane == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(&h_full[s], 1);
            mbar_init(&h_empty[s], 1);
        }
        for (int s = 0; s < SW; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tmem_full[b], 1);
            mbar_init(&tmem_empty[b], 8);   // one arrival per epilogue warp
        }
        mbar_init(mma_done, 1);
        fence_mbar_init();
        tma_prefetch_desc(&maps.a);
        tma_prefetch_desc(&maps.b);
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 8) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t ih = 0, iw = 0;
            bool alive = true;
            for (int t = blockIdx.x; t < p.num_tiles && alive; t += gridDim.x) {
                int n, h0, w0;
                halo_tile(p, t, n, h0, w0);
                for (int c = 0; c < p.chunks && alive; ++c) {
                    const uint32_t sa = ih % SA;
                    if (!mbar_wait_bounded(&h_empty[sa], ((ih / SA) & 1) ^ 1, p.status, DEV_FLAG_WAIT_PRODUCER)) {
                        alive = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&h_full[sa], h_bytes);
                    tma_load_4d(sH + sa * HALO_F_A_BYTES, &maps.a, c * TC_BK, w0 - 1, h0 - 1, n, &h_full[sa]);
                    ++ih;
                    for (int tap = 0; tap < 9; ++tap) {
                        const uint32_t sw = iw % SW;
                        if (!mbar_wait_bounded(&w_empty[sw], ((iw / SW) & 1) ^ 1, p.status, DEV_FLAG_WAIT_PRODUCER)) {
                            alive = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&w_full[sw], HALO_F_W_STAGE);
                        if (p.b_tap_outer)
                            tma_load_3d(sW + sw * HALO_F_W_STAGE, &maps.b, c * TC_BK, 0, tap, &w_full[sw]);
                        else
                            tma_load_3d(sW + sw * HALO_F_W_STAGE, &maps.b, c * TC_BK, tap, 0, &w_full[sw]);
                        ++iw;
                    }
                }
            }
            // every copy issued above has landed before the CTA may exit
            for (uint32_t k = ih > static_cast<uint32_t>(SA) ? ih - SA : 0u; k < ih; ++k)
                if (!mbar_wait_bounded(&h_full[k % SA], (k / SA) & 1, p.status, DEV_FLAG_WAIT_PRODUCER)) break;
            for (uint32_t k = iw > static_cast<uint32_t>(SW) ? iw - SW : 0u; k < iw; ++k)
                if (!mbar_wait_bounded(&w_full[k % SW], (k / SW) & 1, p.status, DEV_FLAG_WAIT_PRODUCER)) break;
        }
        __syncwarp();
    } else if (warp == 9) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t ih = 0, iw = 0, j = 0;
            bool alive = true;
            for (int t = blockIdx.x; t < p.num_tiles && alive; t += gridDim.x, ++j) {
                const uint32_t b = j & 1, tph = (j >> 1) & 1;
                if (!mbar_wait_bounded(&tmem_empty[b], tph ^ 1, p.status, DEV_FLAG_WAIT_MMA)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * ACC_STRIDE;
                for (int c = 0; c < p.chunks && alive; ++c) {
                    const uint32_t sa = ih % SA;
                    if (!mbar_wait_bounded(&h_full[sa], (ih / SA) & 1, p.status, DEV_FLAG_WAIT_MMA)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t h_base = smem_u32(sH + sa * HALO_F_A_BYTES);
                    for (int tap = 0; tap < 9; ++tap) {
                        const uint32_t sw = iw % SW;
                        if (!mbar_wait_bounded(&w_full[sw], (iw / SW) & 1, p.status, DEV_FLAG_WAIT_MMA)) {
                            alive = false;
                            break;
                        }
                        tc_fence_after();
                        const int dh = tap / 3, dw = tap % 3;
                        const int off = p.tap_sign > 0 ? dh * pitch + dw : (2 - dh) * pitch + (2 - dw);
                        const uint32_t b_win = h_base + static_cast<uint32_t>(off) * 128u;
                        const uint32_t a_base = smem_u32(sW + sw * HALO_F_W_STAGE);
#pragma unroll
                        for (int kk = 0; kk < TC_BK / 8; ++kk) {
                            const uint64_t da = smem_desc_sw128(a_base + kk * 32, 16, 1024);
                            const uint64_t db = smem_desc_sw128(b_win + kk * 32, 16, 1024);
                            mma_tf32(d_tmem, da, db, IDESC, (c > 0 || tap > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&w_empty[sw]);
                        ++iw;
                    }
                    if (!alive) break;
                    mma_commit(&h_empty[sa]);
                    ++ih;
                }
                mma_commit(&tmem_full[b]);
            }
            mma_commit(mma_done);
            mbar_wait_bounded(mma_done, 0, p.status, DEV_FLAG_WAIT_MMA);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue (warps 0-7)
        const int quarter = warp & 3, grp = warp >> 2;
        const int co = quarter * 32 + lane;   // this lane's output channel (TMEM lane)
        const bool masked = p.epi == EPI_MASK && p.mask;
        const float bias_co = (p.epi == EPI_STORE && p.bias) ? p.bias[co] : 0.f;
        uint32_t j = 0;
        for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++j) {
            int n, h0, w0;
            halo_tile(p, t, n, h0, w0);
            if (masked) {   // this warp's mask lines (position lane of each of its chunks) on their way to L2
#pragma unroll
                for (int k = 0; k < HALO_F_POS / 64; ++k) {
                    const int pos = (grp + 2 * k) * 32 + lane, hr = pos / pitch, wc = pos - hr * pitch;
                    if (hr < p.bh && wc < p.bw && h0 + hr < p.out_h && w0 + wc < p.out_w)
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(
                            p.mask + ((static_cast<long long>(n) * p.out_h + h0 + hr) * p.out_w + w0 + wc) * p.ldm +
                            quarter * 32)
                                     : "memory");
                }
            }
            const uint32_t b = j & 1, tph = (j >> 1) & 1;
            if (!mbar_wait_bounded(&tmem_full[b], tph, p.status, DEV_FLAG_WAIT_EPILOGUE)) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + b * ACC_STRIDE + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
            for (int k = 0; k < HALO_F_POS / 64; ++k) {
                const int chunk = grp + 2 * k;   // positions 32 chunk .. + 31
                uint32_t v[32];
                __syncwarp();
                tmem_ld_32x32b_x32(tb + chunk * 32, v);
                tmem_wait_ld();
                if (k == HALO_F_POS / 64 - 1) {   // this warp's part of the accumulator is read
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(smem_u32(&tmem_empty[b]));
                }
                // position -> (row, column) of the tile, stepped along the chunk (warp-uniform)
                int hr = (chunk * 32) / pitch, wc = chunk * 32 - hr * pitch;
                long long pix = (static_cast<long long>(n) * p.out_h + h0 + hr) * p.out_w + w0 + wc;
                float mv[32];
                if (masked) {   // the chunk's mask values, all in flight before they are used
                    int hr2 = hr, wc2 = wc;
                    long long px2 = pix;
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const bool ok = hr2 < p.bh && wc2 < p.bw && h0 + hr2 < p.out_h && w0 + wc2 < p.out_w &&
                                        n < p.img_n;
                        mv[q] = ok ? p.mask[px2 * p.ldm + co] : 0.f;
                        if (++wc2 == pitch) {
                            wc2 = 0;
                            ++hr2;
                            px2 += p.out_w - pitch + 1;
                        } else {
                            ++px2;
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const bool ok = hr < p.bh && wc < p.bw && h0 + hr < p.out_h && w0 + wc < p.out_w && n < p.img_n;
                    if (ok) {
                        float x = __uint_as_float(v[q]);
                        if (p.epi == EPI_STORE) {
                            x += bias_co;
                            if (p.relu) x = fmaxf(x, 0.f);
                        } else if (masked) {
                            x = mv[q] > 0.f ? x : 0.f;
                        }
                        p.D[pix * p.ldd + co] = x;
                    }
                    if (++wc == pitch) {
                        wc = 0;
                        ++hr;
                        pix += p.out_w - pitch + 1;
                    } else {
                        ++pix;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

#endif  // __CUDACC__

}  // namespace sprint
