// us_tc.cu -- tensor-core (tcgen05) bitmap SpMM for many tokens (prefill).
//
// Y = W . X, W fp16 stored as 64-column bitmap tiles (IE-BME of "UnionSparse:
// An Index-Efficient Sparsity Framework for Low-Bit Sparse LLM Inference on
// Edge", section V-A, one area, row-major scan), X fp16 token-major, fp32
// accumulation.  Once a tile is decoded it is a dense contraction, so it runs
// on the 5th-generation tensor cores: the prefill kernel of "Unified
// Static-Dynamic Pruning for Efficient LLM Inference" (section 4.3) decodes
// tiles into shared memory and re-lays them out for the tensor cores; here the
// decode writes the tensor cores' own K-major 128-byte-swizzled layout directly,
// so no separate alignment pass is needed.
//
// One CTA computes a 128-row x (256 NH)-token output tile over its K slice
// (NH = 1 or 2 halves of 256 tokens; with two, every decoded A tile feeds twice
// as many tokens):
//  * warp 0 (W producer): 1-D bulk copies of both 64-row bands' bitmap words
//    and value runs for chunks of two 64-column K steps (a band's consecutive
//    tiles are contiguous), packed by their real length into a byte ring (up to
//    eight chunks in flight), the next chunk's tile offsets loaded one ahead;
//  * warp 2 (X producer): 2-D TMA tile loads (128-byte swizzle, zero fill past
//    N) of the matching 256 x 64 activation blocks into the B stage, one per
//    token half that holds tokens;
//  * warps 3-18 (decoders), two groups of eight on alternate K steps, so that
//    two steps are decoded at once into three A stages: four threads per weight
//    row, each rebuilding 16 positions of two rows per K step - rank = row base
//    (warp scan of the band's row popcounts) + running popcount, value =
//    run[rank] or 0 - stored as 16-byte chunks at the swizzled positions of the
//    A stage, then a generic->async proxy fence and an arrive on the stage's
//    "A full" barrier (COL tiles: 4 columns x 4 rows per thread, twice);
//  * warp 1 (MMA): allocates 256 NH TMEM columns; one thread issues four
//    tcgen05.mma kind::f16 (M=128, N=256, K=16) per K step and token half, the
//    halves into adjacent 256-column fp32 accumulators, and commits once per
//    K step to that step's "done" barrier, which frees its A and B stages;
//  * warps 3 .. 3+4NH-1 (epilogue): tcgen05.ld the accumulators (one TMEM lane
//    per output row, one warp per lane quarter and token half) and write fp16
//    outputs.  Under split-K the K slices of an output tile form one
//    thread-block cluster: each CTA parks its fp32 partial of one token half in
//    its own shared memory (the operand stages are free by then), and after a
//    cluster barrier every CTA sums its share of the rows over the cluster's
//    partials (distributed shared memory) in fixed slice order and writes
//    fp16; a second barrier keeps the partials alive until all have read them.
#include <cudaTypedefs.h>

#include "us_common.cuh"
#include "us_internal.h"
#include "us_tcgen05.cuh"

namespace {

constexpr int kBM = 128;                 // output rows per CTA (two 64-row bands)
constexpr int kBH = 256;                 // tokens per MMA (one token half)
constexpr int kBK = 64;                  // K per step (one bitmap tile column)
constexpr int kAStages = 3;              // decoded A stages
constexpr int kSD = 6;                   // "MMAs of step q done" barriers (a multiple of the stage counts)
constexpr int kMaxBStages = 3;           // activation stages, at most
constexpr int kC = 2;                    // K steps per raw chunk (one placement, one barrier)
constexpr int kRawSlots = 8;             // raw chunks that may be in flight
constexpr int kGroups = 2;               // decoder groups, on alternate K steps
constexpr int kGroupWarps = 8;           // warps per decoder group
constexpr int kDecWarps = kGroups * kGroupWarps;
constexpr int kThreads = 32 * (3 + kDecWarps);
constexpr int kABytes = kBM * kBK * 2;           // 16 KB
constexpr int kHBytes = kBH * kBK * 2;           // 32 KB per token half
constexpr int kRawBm = 2 * 512;                  // two bands' bitmaps (64x64 tiles)
constexpr int kRawMax = kC * (kRawBm + 2 * 64 * 64 * 2);   // one chunk's raw weights, worst case (34 KB)
constexpr int kHeader = 1024;
constexpr size_t kSmemCap = 232448;              // dynamic shared memory per CTA

// tile shape for NH token halves; the raw ring takes what the stages leave
template <int NH>
struct TcShape {
    static constexpr int kBN = kBH * NH;
    static constexpr int kBStages = NH == 1 ? 3 : 2;
    static constexpr int kBBytes = kHBytes * NH;
    static constexpr size_t kFixed = 1024 + (size_t)kAStages * kABytes + (size_t)kBStages * kBBytes + kHeader;
    static constexpr size_t kRingAll = kSmemCap - kFixed;
    static constexpr int kRing = (int)((kRingAll > 65536 ? 65536 : kRingAll) & ~size_t(15));
    static constexpr size_t kSmem = kFixed + (size_t)kRing;
    static_assert(kRing >= kRawMax, "the raw ring holds a worst-case chunk");
    static_assert(kSmem <= kSmemCap, "shared memory per CTA");
};

struct TcSmem {
    uint64_t raw_full[kRawSlots], raw_empty[kRawSlots];
    uint64_t a_full[kAStages], b_full[kMaxBStages];
    uint64_t sdone[kSD];                 // step q's MMAs finished: its A and B stages are free
    uint64_t done;
    uint32_t tmem_base;
    uint32_t raw_pos[kRawSlots];         // ring offset of the chunk in slot s
    uint32_t raw_vb0[kRawSlots];         // bytes of band 0's value runs in the chunk
    uint32_t raw_off[kRawSlots][2][kC];  // a tile's run start within its band's runs (elements)
    uint32_t raw_len[kRawSlots][2][kC];  // a tile's run length (elements)
    uint32_t issued_w, issued_x;         // K steps whose copies were issued
    uint32_t flag;
};
static_assert(sizeof(TcSmem) <= kHeader, "header");

// 2-D TMA tile load (x = K element, y = token) completing on `bar`
US_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(us::smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(us::smem_addr(bar))
        : "memory");
}

struct TcParams {
    UsKParams p;
    int n_tiles;          // ceil(N / (256 NH))
};

// The largest K split of the tensor-core path: the slices of an output tile
// form one thread-block cluster (portable cluster size).
constexpr int kMaxSplit = 8;

// Split-K reduction of one token half (ntok tokens from n0) inside the
// cluster: every CTA's fp32 partial sits token-major in its own shared memory
// at `part` (part[n * kBM + row]).  This CTA sums the row groups of four
// [rank * 32 / split, (rank + 1) * 32 / split) over the slices in slice order
// (0 + s0 + s1 + ..., as a plain sequential sum) and writes them as fp16.
US_DEV void tc_cluster_reduce(const UsKParams& p, const float* part, int mt, int n0, int ntok) {
    const uint32_t rank = us::cluster_ctarank();
    const int g0 = (int)(rank * 32u / (uint32_t)p.split), g1 = (int)((rank + 1u) * 32u / (uint32_t)p.split);
    const int ng = g1 - g0;
    for (int it = threadIdx.x; it < ntok * ng; it += kThreads) {
        const int n = it / ng, g = g0 + (it - n * ng);
        const uint32_t off = (uint32_t)(n * kBM + 4 * g) * 4u;
        float4 acc = us::ld_cluster_v4f32(us::cluster_map(part, 0) + off);
        for (int sl = 1; sl < p.split; ++sl) {
            const float4 w = us::ld_cluster_v4f32(us::cluster_map(part, (uint32_t)sl) + off);
            acc.x += w.x; acc.y += w.y; acc.z += w.z; acc.w += w.w;
        }
        const uint32_t lo = (uint32_t)us::float_to_half_bits(acc.x) | ((uint32_t)us::float_to_half_bits(acc.y) << 16);
        const uint32_t hi = (uint32_t)us::float_to_half_bits(acc.z) | ((uint32_t)us::float_to_half_bits(acc.w) << 16);
        *reinterpret_cast<uint2*>(p.Y + (int64_t)(n0 + n) * p.M + mt * kBM + 4 * g) = make_uint2(lo, hi);
    }
}

// Each CTA loads its own activation tiles; CTAs of neighbouring row blocks
// read the same tiles, which the L2 serves after the first.
template <int ORDER, int NH>
__global__ void __launch_bounds__(kThreads, 1)
spmm_f16_tc_kernel(const TcParams tp, const __grid_constant__ CUtensorMap xmap) {
    using Sh = TcShape<NH>;
    constexpr int kBN = Sh::kBN, kBStages = Sh::kBStages, kBBytes = Sh::kBBytes, kRing = Sh::kRing;
    const UsKParams& p = tp.p;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled operand tiles
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* a_st = smem;                                   // kAStages x 16 KB
    uint8_t* b_st = a_st + kAStages * kABytes;              // kBStages x 32 NH KB
    uint8_t* ring = b_st + kBStages * kBBytes;              // raw weights of the K steps in flight
    TcSmem& S = *reinterpret_cast<TcSmem*>(ring + kRing);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = blockIdx.x;                              // 128-row block
    const int slice = blockIdx.y % p.split;                 // K slice (cluster rank under split-K)
    const int nt = blockIdx.y / p.split;                    // token tile
    const int kt0 = (int)((int64_t)slice * p.nTK / p.split);
    const int kt1 = (int)((int64_t)(slice + 1) * p.nTK / p.split);
    const int nk = kt1 - kt0;
    const int band0 = mt * 2;                               // two 64-row bands
    // token halves holding at least one token (the last tile may have one)
    const int halves = NH == 1 ? 1 : (nt * kBN + kBH < p.N ? 2 : 1);
    const uint32_t idesc = us::umma_idesc_f16(kBM, kBH);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRawSlots; ++s) {
            us::mbar_init(&S.raw_full[s], 1);
            us::mbar_init(&S.raw_empty[s], kC * kGroupWarps);   // every step of the chunk
        }
        for (int s = 0; s < kAStages; ++s) us::mbar_init(&S.a_full[s], kGroupWarps);
        for (int s = 0; s < kBStages; ++s) us::mbar_init(&S.b_full[s], 1);
        for (int s = 0; s < kSD; ++s) us::mbar_init(&S.sdone[s], 1);
        us::mbar_init(&S.done, 1);
        S.issued_w = S.issued_x = 0;
        us::fence_mbar_init();
    }
    if (warp == 1) us::tmem_alloc(&S.tmem_base, kBN);
    __syncthreads();
    us::tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    us::pdl_wait();
    bool failed = false;

    if (warp == 0) {
        // ------------------------------------------------------- W producer
        // Chunks of kC consecutive K steps: a band's tiles are consecutive in
        // the bitmap and in the value array, so a chunk is four bulk copies
        // (each band's bitmaps, each band's value runs), packed by real length
        // into a byte ring (16-byte aligned).  One thread places and issues;
        // the next chunk's tile offsets are loaded one chunk ahead.  The ring
        // holds the chunks [tail, c) in order, from the start of chunk `tail`
        // to `head`, wrapping at kRing.
        if (lane == 0) {
            const int nch = (nk + kC - 1) / kC;
            uint32_t no[2][kC + 1];
            auto load_offs = [&](int c) {
                const int q0 = c * kC, cnt = min(kC, nk - q0);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int j = 0; j <= kC; ++j)
                        no[h][j] = p.tile_off[(int64_t)(band0 + h) * p.nTK + kt0 + q0 + min(j, cnt)];
            };
            if (nch > 0) load_offs(0);
            uint32_t head = 0;
            int tail = 0;
            for (int c = 0; c < nch; ++c) {
                const int slot = c % kRawSlots, q0 = c * kC, cnt = min(kC, nk - q0);
                uint32_t o[2][kC + 1];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int j = 0; j <= kC; ++j) o[h][j] = no[h][j];
                if (c + 1 < nch) load_offs(c + 1);
                uint32_t vb[2];
                bool good[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    good[h] = (o[h][0] & 7u) == 0 && (uint64_t)o[h][kC] * 2u <= p.values_bytes;
#pragma unroll
                    for (int j = 0; j < kC; ++j)
                        good[h] = good[h] && o[h][j + 1] >= o[h][j] && (o[h][j + 1] - o[h][j]) <= 4096u &&
                                  (o[h][j + 1] & 7u) == 0;
                    vb[h] = good[h] ? (o[h][kC] - o[h][0]) * 2u : 0u;
                }
                const uint32_t sz = (uint32_t)cnt * kRawBm + vb[0] + vb[1];
                uint32_t place = 0;
                bool fail = false;
                for (;;) {
                    const int inflight = c - tail;
                    if (inflight == 0) { place = 0; break; }
                    if (inflight < kRawSlots) {
                        const uint32_t s0 = S.raw_pos[tail % kRawSlots];
                        if (head > s0) {
                            if (head + sz <= (uint32_t)kRing) { place = head; break; }
                            if (sz <= s0) { place = 0; break; }
                        } else if (head + sz <= s0) {
                            place = head;
                            break;
                        }
                    }
                    if (!us::mbar_wait(&S.raw_empty[tail % kRawSlots], (uint32_t)(tail / kRawSlots) & 1u, p.status)) {
                        fail = true;
                        break;
                    }
                    ++tail;
                }
                if (fail) {
                    failed = true;
                    break;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (!good[h]) us::set_status(p.status, US_ERR_CORRUPT);
#pragma unroll
                    for (int j = 0; j < kC; ++j) {
                        S.raw_off[slot][h][j] = good[h] ? o[h][j] - o[h][0] : 0u;
                        S.raw_len[slot][h][j] = good[h] ? o[h][j + 1] - o[h][j] : 0u;
                    }
                }
                S.raw_vb0[slot] = vb[0];
                S.raw_pos[slot] = place;
                uint8_t* r = ring + place;
                us::mbar_arrive_expect_tx(&S.raw_full[slot], sz);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int64_t t = (int64_t)(band0 + h) * p.nTK + kt0 + q0;
                    us::bulk_g2s(r + h * cnt * 512, p.bitmap + t * 64, (uint32_t)cnt * 512u, &S.raw_full[slot]);
                    if (vb[h])
                        us::bulk_g2s(r + 2 * cnt * 512 + (h ? vb[0] : 0u), p.values + (uint64_t)o[h][0] * 2u, vb[h],
                                     &S.raw_full[slot]);
                }
                // a short last chunk: arrive for the steps it does not have
                if (cnt < kC) us::mbar_arrive_n(&S.raw_empty[slot], (uint32_t)((kC - cnt) * kGroupWarps));
                head = place + sz;
                S.issued_w = (uint32_t)(c + 1);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------- X producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
            for (int q = 0; q < nk; ++q) {
                const int s = q % kBStages;
                if (q >= kBStages &&
                    !us::mbar_wait(&S.sdone[(q - kBStages) % kSD], ((q - kBStages) / kSD) & 1, p.status)) {
                    failed = true;
                    break;
                }
                us::mbar_arrive_expect_tx(&S.b_full[s], (uint32_t)(kHBytes * halves));
                for (int h = 0; h < halves; ++h)
                    tma_load_2d(b_st + s * kBBytes + h * kHBytes, &xmap, (kt0 + q) * kBK, nt * kBN + h * kBH,
                                &S.b_full[s]);
                S.issued_x = (uint32_t)(q + 1);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            for (int q = 0; q < nk; ++q) {
                const int sa = q % kAStages, sb = q % kBStages;
                if (!us::mbar_wait(&S.a_full[sa], (q / kAStages) & 1, p.status) ||
                    !us::mbar_wait(&S.b_full[sb], (q / kBStages) & 1, p.status)) {
                    failed = true;
                    break;
                }
                us::tc_fence_after();
                const uint64_t ad = us::umma_smem_desc_sw128(a_st + sa * kABytes);
                const uint64_t bd = us::umma_smem_desc_sw128(b_st + sb * kBBytes);
                // K = 16 per MMA: +32 bytes = +2 in the descriptor's address field;
                // token half h: +32 KB of B, +256 TMEM columns
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    for (int h = 0; h < halves; ++h)
                        us::umma_f16(tmem + (uint32_t)(h * kBH), ad + 2 * kk, bd + (uint64_t)(h * (kHBytes >> 4)) + 2 * kk,
                                     idesc, (q > 0 || kk > 0) ? 1u : 0u);
                // one release for both stages
                us::umma_commit(&S.sdone[q % kSD]);
            }
            us::umma_commit(&S.done);
        }
    } else {
        // ------------------------------------------------------------ decoders
        // two groups of eight warps take alternate K steps, so two steps are
        // decoded at once while the tensor core works on an earlier one; a warp
        // covers 16 rows of the 128-row A tile
        const int d = warp - 3;
        const int grp = d / kGroupWarps, dd = d % kGroupWarps;
        const int band_h = dd >> 2;                        // 16 dd .. 16 dd + 15 lie in one band
        for (int q = grp; q < nk; q += kGroups) {
            const int ch = q / kC, jj = q % kC, slot = ch % kRawSlots, sa = q % kAStages;
            const int cnt = min(kC, nk - ch * kC);
            if (!us::mbar_wait(&S.raw_full[slot], (ch / kRawSlots) & 1, p.status)) {
                failed = true;
                break;
            }
            const uint8_t* r = ring + S.raw_pos[slot];
            const uint64_t* bm = reinterpret_cast<const uint64_t*>(r + (band_h * cnt + jj) * 512);
            // bases: popcounts of the earlier rows (ROW) or columns (COL) of the
            // band, one warp scan of packed pairs
            const uint64_t w0 = bm[lane], w1 = bm[lane + 32];
            const uint32_t packed = (uint32_t)__popcll(w0) | ((uint32_t)__popcll(w1) << 16);
            uint32_t incl = packed;
#pragma unroll
            for (int sh = 1; sh < 32; sh <<= 1) {
                const uint32_t o = __shfl_up_sync(0xffffffffu, incl, sh);
                if (lane >= sh) incl += o;
            }
            const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
            const uint32_t ex = incl - packed;
            const uint32_t P = (tot & 0xFFFFu) + (tot >> 16);
            const bool ok = P <= S.raw_len[slot][band_h][jj];
            if (!ok && lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
            const uint16_t* run = reinterpret_cast<const uint16_t*>(
                r + 2 * cnt * 512 + (band_h ? S.raw_vb0[slot] : 0u) + S.raw_off[slot][band_h][jj] * 2u);
            if constexpr (ORDER == US_ORDER_ROW) {
                // four threads per row (16 positions each), rows i and i + 8:
                // rank = row base + running popcount, value = run[rank] or 0,
                // stored as 16-byte chunks at their swizzled place
                const int qq = lane & 3;
                uint32_t bits[2], rank[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int ib = ((16 * dd) & 63) + (lane >> 2) + 8 * u;      // row within the band
                    const uint32_t exr = __shfl_sync(0xffffffffu, ex, ib & 31);
                    const uint32_t rowbase = (ib < 32) ? (exr & 0xFFFFu) : (tot & 0xFFFFu) + (exr >> 16);
                    const uint64_t word = bm[ib];
                    bits[u] = ok ? (uint32_t)(word >> (16 * qq)) & 0xFFFFu : 0u;
                    rank[u] = rowbase + (uint32_t)__popcll(word & ((1ull << (16 * qq)) - 1ull));
                }
                // wait for the A stage to be free (the MMA of step q - kAStages finished)
                if (q >= kAStages &&
                    !us::mbar_wait(&S.sdone[(q - kAStages) % kSD], ((q - kAStages) / kSD) & 1, p.status)) {
                    failed = true;
                    break;
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int row = 16 * dd + (lane >> 2) + 8 * u;    // row & 7 == lane >> 2
                    uint8_t* arow = a_st + sa * kABytes + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {                 // 8 positions per 16-byte chunk
                        uint32_t h2[4];
#pragma unroll
                        for (int j = 0; j < 8; j += 2) {
                            const uint32_t b0 = (bits[u] >> (8 * c + j)) & 1u;
                            const uint32_t b1 = (bits[u] >> (8 * c + j + 1)) & 1u;
                            const uint32_t v0 = b0 ? run[rank[u]] : 0u;
                            rank[u] += b0;
                            const uint32_t v1 = b1 ? run[rank[u]] : 0u;
                            rank[u] += b1;
                            h2[j >> 1] = v0 | (v1 << 16);
                        }
                        const int chunk = 2 * qq + c;
                        *reinterpret_cast<uint4*>(arow + ((chunk ^ (row & 7)) << 4)) =
                            make_uint4(h2[0], h2[1], h2[2], h2[3]);
                    }
                }
            } else {
                // COL tiles (Tiled-CBC of "Unified Static-Dynamic Pruning for
                // Efficient LLM Inference", section 4.1: one bitmap word per
                // column, the values column after column).  A thread rebuilds 4
                // adjacent columns x 4 rows, twice (row groups rg and rg + 2): per
                // column, rank = column base + popcount of the rows above +
                // running count; per row it stores the 4 values as one 8-byte
                // piece of the K-major swizzled A stage - the layout alignment of
                // that page's section 4.3 done by the decoder's own stores.
                const int quad = lane & 15;                    // columns 4 quad .. 4 quad + 3
                uint32_t base[4];
                uint64_t wc[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = 4 * quad + c;
                    const uint32_t e = __shfl_sync(0xffffffffu, ex, j & 31);
                    base[c] = j < 32 ? (e & 0xFFFFu) : (tot & 0xFFFFu) + (e >> 16);
                    wc[c] = ok ? bm[j] : 0ull;
                }
                if (q >= kAStages &&
                    !us::mbar_wait(&S.sdone[(q - kAStages) % kSD], ((q - kAStages) / kSD) & 1, p.status)) {
                    failed = true;
                    break;
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int rg = 4 * (dd & 3) + (lane >> 4) + 2 * u;    // rows 4 rg .. 4 rg + 3 of the band
                    const uint64_t below = rg ? (~0ull >> (64 - 4 * rg)) : 0ull;
                    uint32_t bits[4], rank[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        rank[c] = base[c] + (uint32_t)__popcll(wc[c] & below);
                        bits[c] = (uint32_t)(wc[c] >> (4 * rg)) & 0xFu;
                    }
                    // row m = 64 band_h + 4 rg + i: 128 bytes at m * 128, chunk
                    // (4 quad >> 3) ^ (m & 7), half (quad & 1) of it
                    uint8_t* arow = a_st + sa * kABytes + (64 * band_h + 4 * rg) * 128 + (quad & 1) * 8;
                    const int m7 = 4 * (rg & 1);               // (m & 7) - i
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t v[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint32_t bb = (bits[c] >> i) & 1u;
                            v[c] = bb ? run[rank[c]] : 0u;
                            rank[c] += bb;
                        }
                        *reinterpret_cast<uint2*>(arow + i * 128 + (((quad >> 1) ^ (m7 + i)) << 4)) =
                            make_uint2(v[0] | (v[1] << 16), v[2] | (v[3] << 16));
                    }
                }
            }
            us::fence_proxy_async_smem();                  // generic writes -> visible to the tensor core
            __syncwarp();
            if (lane == 0) {
                us::mbar_arrive(&S.a_full[sa]);
                us::mbar_arrive(&S.raw_empty[slot]);
            }
        }
    }

    // ---------------------------------------------------------------- epilogue
    __syncthreads();
    const bool any_failed = __syncthreads_or(failed);
    if (any_failed && warp == 0 && lane == 0) {
        // let this CTA's copies still in flight land (bounded) before it exits:
        // the last issued step of each slot / stage
        const int iw = (int)S.issued_w, ix = (int)S.issued_x;
        for (int c = iw > kRawSlots ? iw - kRawSlots : 0; c < iw; ++c)
            us::mbar_wait(&S.raw_full[c % kRawSlots], (c / kRawSlots) & 1, nullptr);
        for (int q = ix > kBStages ? ix - kBStages : 0; q < ix; ++q)
            us::mbar_wait(&S.b_full[q % kBStages], (q / kBStages) & 1, nullptr);
    }
    bool ready = false;
    if (warp >= 3 && warp < 3 + 4 * halves) {
        // the final commit also covers MMAs issued before a failure: wait for it (bounded)
        ready = us::mbar_wait(&S.done, 0, any_failed ? nullptr : p.status) && !any_failed;
        us::tc_fence_after();
    }
    const int quarter = warp & 3;                           // TMEM lanes 32*quarter .. +31
    const int m = mt * kBM + quarter * 32 + lane;
    const int nbase = nt * kBN;
    if (p.split == 1) {
        if (warp >= 3 && warp < 3 + 4 * halves) {
            const int half = (warp - 3) >> 2;               // token half: TMEM columns 256 half ..
            for (int c0 = half * kBH; c0 < (half + 1) * kBH && nbase + c0 < p.N; c0 += 32) {
                float v[32];
                us::tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
                if (!ready) continue;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int n = nbase + c0 + i;
                    if (n < p.N) p.Y[(int64_t)n * p.M + m] = us::float_to_half_bits(v[i]);
                }
            }
        }
    } else {
        // split-K inside the cluster, one token half at a time: every thread of
        // every CTA reaches both barriers of every round (the rounds depend on
        // nt only, the same for the whole cluster); a failed CTA writes nothing
        // and its outputs are not valid (the status word says why)
        __syncthreads();                                    // the copies of a failed CTA have landed
        float* part = reinterpret_cast<float*>(smem);       // 128 rows x 256 tokens fp32, token-major
        for (int hh = 0; hh < halves; ++hh) {
            if (warp >= 3 + 4 * hh && warp < 7 + 4 * hh) {
                for (int c0 = 0; c0 < kBH; c0 += 32) {
                    float v[32];
                    us::tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(hh * kBH + c0), v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) part[(c0 + i) * kBM + quarter * 32 + lane] = ready ? v[i] : 0.f;
                }
            }
            us::cluster_sync();
            const int n0 = nbase + hh * kBH;
            if (!any_failed) tc_cluster_reduce(p, part, mt, n0, min(kBH, p.N - n0));
            us::cluster_sync();                             // the partials stay until every CTA has read them
        }
    }
    us::tc_fence_before();
    __syncthreads();
    if (warp == 1) us::tmem_dealloc(tmem, kBN);
}

}  // namespace

namespace us {

// the driver's tiled tensor-map encoder, looked up once
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

bool tc_f16_supported(int TM, int TK, int M, int N) {
    return TM == 64 && TK == 64 && M % kBM == 0 && N >= 64;
}

// 512 tokens per CTA once there are more than 256: each decoded A tile then
// feeds twice as many tokens
int tc_tok_block(int N) { return N > kBH ? 2 * kBH : kBH; }

int tc_split(int M, int N, int nTK) {
    const int bn = tc_tok_block(N);
    const int ctas = (M / kBM) * ((N + bn - 1) / bn);
    int s = 1;
    while (ctas * s * 2 <= num_sms() && nTK / (s * 2) >= 8 && s < kMaxSplit) s *= 2;
    return s;
}

int tc_max_split() { return kMaxSplit; }

// The split-K partials stay in the cluster's shared memory: no workspace.
size_t tc_ws(int, int, int) { return 0; }

us_status launch_tc_f16(const UsKParams& p, cudaStream_t st) {
    auto enc = tensor_map_encoder();
    if (!enc) return US_ERR_CUDA;
    if (p.tok_block != kBH && p.tok_block != 2 * kBH) return US_ERR_INVALID_ARG;
    const bool two = p.tok_block == 2 * kBH;
    CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)p.K, (cuuint64_t)p.N};
    const cuuint64_t gstride[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBH};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(p.X), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return US_ERR_CUDA;
    TcParams tp;
    tp.p = p;
    tp.n_tiles = (p.N + p.tok_block - 1) / p.tok_block;
    const bool col = p.order == US_ORDER_COL;
    void (*kern)(const TcParams, const CUtensorMap) =
        two ? (col ? spmm_f16_tc_kernel<US_ORDER_COL, 2> : spmm_f16_tc_kernel<US_ORDER_ROW, 2>)
            : (col ? spmm_f16_tc_kernel<US_ORDER_COL, 1> : spmm_f16_tc_kernel<US_ORDER_ROW, 1>);
    const size_t smem = two ? TcShape<2>::kSmem : TcShape<1>::kSmem;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return US_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    if (p.split < 1 || p.split > kMaxSplit) return US_ERR_INVALID_ARG;
    cfg.gridDim = dim3((unsigned)(p.M / kBM), (unsigned)(tp.n_tiles * p.split));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    // the K slices of an output tile (consecutive blockIdx.y) form one cluster
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)p.split;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.split > 1 ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, tp, map) != cudaSuccess) return US_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? US_OK : US_ERR_CUDA;
}

}  // namespace us
