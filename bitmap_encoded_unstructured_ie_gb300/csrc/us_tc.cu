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
// One CTA computes a 128-row x 256-token output tile over its K slice:
//  * warp 0 (producer): 1-D bulk copies of both 64-row bands' bitmap words and
//    value runs for each 64-column K step into a raw ring, and a 2-D TMA tile
//    load (128-byte swizzle, zero fill past N) of the matching 256 x 64
//    activation block into the B stage;
//  * warps 2-9 (decoders): two threads per weight row; each rebuilds 32
//    positions per K step - rank = row base (warp scan of the band's row
//    popcounts) + running popcount, value = run[rank] or 0 - and stores them as
//    16-byte chunks at the swizzled positions of the A stage, then fences the
//    generic->async proxy and arrives on the stage's "A full" barrier;
//  * warp 1 (MMA): allocates 256 TMEM columns; one thread issues four
//    tcgen05.mma kind::f16 (M=128, N=256, K=16) per K step with the fp32
//    accumulator in TMEM and commits to the stage's "empty" barrier;
//  * warps 2-5 (epilogue): tcgen05.ld the accumulator (one TMEM lane per
//    output row) and write fp16 outputs, or, under split-K, fp32 partials that
//    the last CTA of the tile sums in fixed slice order.
#include <cudaTypedefs.h>

#include "us_common.cuh"
#include "us_internal.h"

namespace {

constexpr int kBM = 128;                 // output rows per CTA (two 64-row bands)
constexpr int kBN = 256;                 // tokens per CTA
constexpr int kBK = 64;                  // K per step (one bitmap tile column)
constexpr int kStages = 3;               // A/B stages
constexpr int kRawStages = 3;            // raw W staging
constexpr int kDecWarps = 8;
constexpr int kThreads = 32 * (2 + kDecWarps);
constexpr int kABytes = kBM * kBK * 2;           // 16 KB
constexpr int kBBytes = kBN * kBK * 2;           // 32 KB
constexpr int kRawBm = 2 * 512;                  // two bands' bitmaps (64x64 tiles)
constexpr int kRawVal = 2 * 64 * 64 * 2;         // two bands' fp16 runs, worst case
constexpr int kRawBytes = kRawBm + kRawVal;      // 17 KB

struct TcSmem {
    uint64_t raw_full[kRawStages], raw_empty[kRawStages];
    uint64_t a_full[kStages], b_full[kStages], ab_empty[kStages];
    uint64_t done;
    uint32_t tmem_base;
    uint32_t raw_len[kRawStages][2];     // run length (elements) of each band's tile
    uint32_t flag;
};

// ------------------------------------------------------------ tcgen05 PTX --
US_DEV uint64_t umma_smem_desc_sw128(const void* p) {
    // K-major, 128-byte swizzle: start address >> 4, LBO unused (1), SBO = 1024 B
    // (8 rows x 128 B), descriptor version 1, layout type 2 (SWIZZLE_128B).
    const uint64_t addr = (uint64_t)(us::smem_addr(p) >> 4) & 0x3FFFull;
    return addr | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f16 instruction descriptor: D fp32, A/B fp16, both K-major, N>>3, M>>4
constexpr uint32_t umma_idesc_f16(int M, int N) {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

US_DEV void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

US_DEV void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     us::smem_addr(bar))
                 : "memory");
}

US_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(us::smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

US_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

US_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
US_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane (base+i)
US_DEV void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 16 consecutive fp32 columns
US_DEV void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

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
    int n_tiles;          // ceil(N / kBN)
};

__global__ void __launch_bounds__(kThreads, 1)
spmm_f16_tc_kernel(const TcParams tp, const __grid_constant__ CUtensorMap xmap) {
    const UsKParams& p = tp.p;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled operand tiles
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* a_st = smem;                                   // kStages x 16 KB
    uint8_t* b_st = a_st + kStages * kABytes;               // kStages x 32 KB
    uint8_t* raw = b_st + kStages * kBBytes;                // kRawStages x 17 KB
    TcSmem& S = *reinterpret_cast<TcSmem*>(raw + kRawStages * kRawBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = blockIdx.x;                              // 128-row block
    const int nt = blockIdx.y % tp.n_tiles;                 // token tile
    const int slice = blockIdx.y / tp.n_tiles;              // K slice
    const int kt0 = (int)((int64_t)slice * p.nTK / p.split);
    const int kt1 = (int)((int64_t)(slice + 1) * p.nTK / p.split);
    const int nk = kt1 - kt0;
    const int band0 = mt * 2;                               // two 64-row bands
    const uint32_t idesc = umma_idesc_f16(kBM, kBN);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRawStages; ++s) {
            us::mbar_init(&S.raw_full[s], 1);
            us::mbar_init(&S.raw_empty[s], kDecWarps);
        }
        for (int s = 0; s < kStages; ++s) {
            us::mbar_init(&S.a_full[s], kDecWarps);
            us::mbar_init(&S.b_full[s], 1);
            us::mbar_init(&S.ab_empty[s], 1);
        }
        us::mbar_init(&S.done, 1);
        us::fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&S.tmem_base, kBN);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    us::pdl_wait();
    bool failed = false;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
            for (int q = 0; q < nk && !failed; ++q) {
                const int rs = q % kRawStages, s = q % kStages;
                if (q >= kRawStages && !us::mbar_wait(&S.raw_empty[rs], ((q / kRawStages) - 1) & 1, p.status)) {
                    failed = true;
                    break;
                }
                uint32_t vb[2], o0[2];
                for (int h = 0; h < 2; ++h) {
                    const int64_t t = (int64_t)(band0 + h) * p.nTK + kt0 + q;
                    const uint32_t a = p.tile_off[t], b = p.tile_off[t + 1];
                    const bool ok = b >= a && (b - a) <= 4096u && (a & 7u) == 0 && (b & 7u) == 0 &&
                                    (uint64_t)b * 2u <= p.values_bytes;
                    if (!ok) us::set_status(p.status, US_ERR_CORRUPT);
                    o0[h] = a;
                    vb[h] = ok ? (b - a) * 2u : 0u;
                    S.raw_len[rs][h] = ok ? (b - a) : 0u;
                }
                uint8_t* r = raw + rs * kRawBytes;
                us::mbar_arrive_expect_tx(&S.raw_full[rs], kRawBm + vb[0] + vb[1]);
                for (int h = 0; h < 2; ++h) {
                    const int64_t t = (int64_t)(band0 + h) * p.nTK + kt0 + q;
                    us::bulk_g2s(r + h * 512, p.bitmap + t * 64, 512, &S.raw_full[rs]);
                    if (vb[h]) us::bulk_g2s(r + kRawBm + h * 8192, p.values + (uint64_t)o0[h] * 2u, vb[h], &S.raw_full[rs]);
                }
                // activation tile for this K step
                if (q >= kStages && !us::mbar_wait(&S.ab_empty[s], ((q / kStages) - 1) & 1, p.status)) {
                    failed = true;
                    break;
                }
                us::mbar_arrive_expect_tx(&S.b_full[s], kBBytes);
                tma_load_2d(b_st + s * kBBytes, &xmap, (kt0 + q) * kBK, nt * kBN, &S.b_full[s]);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            for (int q = 0; q < nk; ++q) {
                const int s = q % kStages;
                if (!us::mbar_wait(&S.a_full[s], (q / kStages) & 1, p.status) ||
                    !us::mbar_wait(&S.b_full[s], (q / kStages) & 1, p.status)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = umma_smem_desc_sw128(a_st + s * kABytes);
                const uint64_t bd = umma_smem_desc_sw128(b_st + s * kBBytes);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)   // K = 16 per MMA: +32 bytes = +2 in the address field
                    umma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (q > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&S.ab_empty[s]);
            }
            umma_commit(&S.done);
        }
    } else {
        // ------------------------------------------------------------ decoders
        const int d = warp - 2;                            // 0..7: rows 16d .. 16d+15
        const int row = 16 * d + (lane >> 1);              // 0..127 within the block
        const int hb = lane & 1;                           // which 32 positions of the row
        const int band_h = row >> 6, i_in_band = row & 63;
        for (int q = 0; q < nk; ++q) {
            const int rs = q % kRawStages, s = q % kStages;
            if (!us::mbar_wait(&S.raw_full[rs], (q / kRawStages) & 1, p.status)) {
                failed = true;
                break;
            }
            const uint8_t* r = raw + rs * kRawBytes;
            const uint64_t* bm = reinterpret_cast<const uint64_t*>(r + band_h * 512);
            // row base: popcounts of the earlier rows of this band (warp scan)
            const uint64_t w0 = bm[lane], w1 = bm[lane + 32];
            const uint32_t packed = (uint32_t)__popcll(w0) | ((uint32_t)__popcll(w1) << 16);
            uint32_t incl = packed;
#pragma unroll
            for (int dd = 1; dd < 32; dd <<= 1) {
                const uint32_t o = __shfl_up_sync(0xffffffffu, incl, dd);
                if (lane >= dd) incl += o;
            }
            const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
            const uint32_t ex = incl - packed;
            const uint32_t exr = __shfl_sync(0xffffffffu, ex, i_in_band & 31);
            const uint32_t rowbase = (i_in_band < 32) ? (exr & 0xFFFFu) : (tot & 0xFFFFu) + (exr >> 16);
            const uint32_t P = (tot & 0xFFFFu) + (tot >> 16);
            const bool ok = P <= S.raw_len[rs][band_h];
            if (!ok && lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
            const uint64_t word = bm[i_in_band];
            const uint32_t bits = hb ? (uint32_t)(word >> 32) : (uint32_t)word;
            uint32_t rank = rowbase + (hb ? (uint32_t)__popc((uint32_t)word) : 0u);
            const uint16_t* run = reinterpret_cast<const uint16_t*>(r + kRawBm + band_h * 8192);
            // wait for the A stage to be free (the MMA of step q - kStages finished)
            if (q >= kStages && !us::mbar_wait(&S.ab_empty[s], ((q / kStages) - 1) & 1, p.status)) {
                failed = true;
                break;
            }
            uint8_t* arow = a_st + s * kABytes + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {                  // 8 positions per 16-byte chunk
                uint32_t h2[4];
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    const uint32_t b0 = ok ? (bits >> (8 * c + j)) & 1u : 0u;
                    const uint32_t b1 = ok ? (bits >> (8 * c + j + 1)) & 1u : 0u;
                    const uint32_t v0 = b0 ? run[rank] : 0u;
                    rank += b0;
                    const uint32_t v1 = b1 ? run[rank] : 0u;
                    rank += b1;
                    h2[j >> 1] = v0 | (v1 << 16);
                }
                const int chunk = 4 * hb + c;
                *reinterpret_cast<uint4*>(arow + ((chunk ^ (row & 7)) << 4)) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
            }
            us::fence_proxy_async_smem();                  // generic writes -> visible to the tensor core
            __syncwarp();
            if (lane == 0) {
                us::mbar_arrive(&S.a_full[s]);
                us::mbar_arrive(&S.raw_empty[rs]);
            }
        }
    }

    // ---------------------------------------------------------------- epilogue
    __syncthreads();
    const bool any_failed = __syncthreads_or(failed);
    if (any_failed && warp == 0 && lane == 0) {
        // let this CTA's copies still in flight land (bounded) before it exits
        for (int q = nk > kRawStages ? nk - kRawStages : 0; q < nk; ++q)
            us::mbar_wait(&S.raw_full[q % kRawStages], (q / kRawStages) & 1, nullptr);
        for (int q = nk > kStages ? nk - kStages : 0; q < nk; ++q)
            us::mbar_wait(&S.b_full[q % kStages], (q / kStages) & 1, nullptr);
    }
    if (warp >= 2 && warp < 6) {
        // the final commit also covers MMAs issued before a failure: wait for it (bounded)
        const bool ready = us::mbar_wait(&S.done, 0, any_failed ? nullptr : p.status) && !any_failed;
        tc_fence_after();
        const int quarter = warp & 3;                       // TMEM lanes 32*quarter .. +31
        const int m = mt * kBM + quarter * 32 + lane;
        const int nbase = nt * kBN;
        float* part = reinterpret_cast<float*>(p.ws);
        const int nTB = tp.n_tiles;
        for (int c0 = 0; c0 < kBN; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
            if (!ready) continue;
            if (p.split > 1) {
                const int64_t base = (((int64_t)slice * nTB + nt) * p.M + m) * kBN + c0;
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    __stcg(reinterpret_cast<float4*>(part + base + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int n = nbase + c0 + i;
                    if (n < p.N) p.Y[(int64_t)n * p.M + m] = us::float_to_half_bits(v[i]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, kBN);
    if (p.split > 1 && !any_failed) {
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0)
            S.flag = (atomicAdd(&p.counters[mt * tp.n_tiles + nt], 1u) == (unsigned)p.split - 1u) ? 1u : 0u;
        __syncthreads();
        if (!S.flag) return;
        __threadfence();
        // the last CTA of this output tile: sum the slices in order, leave zeros behind
        float* part = reinterpret_cast<float*>(p.ws);
        for (int idx = threadIdx.x; idx < kBM * kBN; idx += kThreads) {
            const int mr = idx / kBN, nc = idx - mr * kBN;
            const int m = mt * kBM + mr, n = nt * kBN + nc;
            float acc = 0.f;
            for (int sl = 0; sl < p.split; ++sl) {
                float* src = part + (((int64_t)sl * tp.n_tiles + nt) * p.M + m) * kBN + nc;
                acc += __ldcg(src);
                __stcg(src, 0.f);
            }
            if (n < p.N) p.Y[(int64_t)n * p.M + m] = us::float_to_half_bits(acc);
        }
        if (threadIdx.x == 0) p.counters[mt * tp.n_tiles + nt] = 0u;
    }
}

// ============================================================== W4A4 path ==
// W4A4 with 8..32 tokens on the tensor cores: the decode is paid once per
// weight position whatever N is.  int4 codes become exact fp16 values (the
// fp16 bit pattern 0x6400 | (w + 8) is 1024 + w + 8; subtracting 1032 leaves w),
// products of |w|, |x| <= 8 are exact, and fp32 accumulation of such integers
// is exact below 2^24, so the int32 results match the integer definition.
//
// One CTA: 128 weight rows (two 64-row bands) x all tokens (padded to BN = 16
// or 32) over its K slice; the K slices of a 128-row block form one cluster.
//  * warp 0: bulk copies of the CTA's packed activations (once) and, per K
//    step, of both bands' bitmaps and nibble runs into a raw ring;
//  * warps 2-9: two threads per weight row decode 32 positions each per K step
//    (byte-steps as in the CUDA-core kernel, emitting fp16) into the swizzled
//    K-major A stage, and convert the K step's activations into the B stage;
//  * warp 1: 4 x tcgen05.mma kind::f16 (M=128, N=BN, K=16) per K step, fp32 in
//    TMEM;
//  * epilogue: TMEM -> int32 in shared memory -> sum over the cluster's slices
//    through distributed shared memory -> Yacc and the dequantised fp16 Y.
constexpr int kW4Stages = 2;
constexpr int kW4Chunk = 4;                            // K steps per bulk-copy chunk
constexpr int kW4BmBand = kW4Chunk * 512;              // one band's bitmaps in a chunk
constexpr int kW4ValBand = kW4Chunk * 2048;            // one band's runs in a chunk (worst case)
constexpr int kW4ChunkBytes = 2 * kW4BmBand + 2 * kW4ValBand;   // 20 KB
constexpr int kW4Dec = 8;
constexpr int kW4Threads = 32 * (2 + kW4Dec);
constexpr int kW4LutRep = 16;

struct W4Smem {
    uint64_t chunk_full[2], chunk_empty[2];
    uint64_t a_full[kW4Stages], ab_empty[kW4Stages];
    uint64_t x_full, done;
    uint32_t tmem_base;
    uint32_t chunk_bad[2];
};

__device__ __forceinline__ uint4 i4x8_to_f16x8(uint32_t even, uint32_t odd, uint32_t sel) {
    // even/odd: bytes (w + 8) of ranks 0,2,4,6 / 1,3,5,7 (rank 7 byte = 8 when unset)
    const uint32_t d0 = __byte_perm(even, odd, sel);
    const uint32_t d1 = __byte_perm(even, odd, sel >> 16);
    const uint32_t k64 = 0x64646464u;
    __half2 h[4];
    const uint32_t b[4] = {__byte_perm(d0, k64, 0x5140), __byte_perm(d0, k64, 0x7362),
                           __byte_perm(d1, k64, 0x5140), __byte_perm(d1, k64, 0x7362)};
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __hsub2(*reinterpret_cast<const __half2*>(&b[i]), bias);
    return make_uint4(*reinterpret_cast<uint32_t*>(&h[0]), *reinterpret_cast<uint32_t*>(&h[1]),
                      *reinterpret_cast<uint32_t*>(&h[2]), *reinterpret_cast<uint32_t*>(&h[3]));
}

template <int BN>
__global__ void __launch_bounds__(kW4Threads, 1)
w4a4_tc_kernel(const UsKParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int kA = kBM * kBK * 2;                       // 16 KB
    constexpr int kB = BN * kBK * 2;                        // 2 or 4 KB
    uint8_t* a_st = smem;
    uint8_t* b_st = a_st + kW4Stages * kA;
    uint8_t* chunks = b_st + kW4Stages * kB;                // 2 x 20 KB
    uint32_t* lut = reinterpret_cast<uint32_t*>(chunks + 2 * kW4ChunkBytes);
    W4Smem& S = *reinterpret_cast<W4Smem*>(lut + 256 * kW4LutRep);
    uint32_t* offs = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(&S) + ((sizeof(W4Smem) + 127) & ~size_t(127)));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = blockIdx.x / p.split;                    // 128-row block; its K slices form a cluster
    const int slice = blockIdx.x % p.split;
    const int kt0 = (int)((int64_t)slice * p.nTK / p.split);
    const int kt1 = (int)((int64_t)(slice + 1) * p.nTK / p.split);
    const int nk = kt1 - kt0;
    const int nchunks = (nk + kW4Chunk - 1) / kW4Chunk;
    const int ostride = (nk + 1 + 3) & ~3;                  // offs[h * ostride + q]
    uint8_t* xs = reinterpret_cast<uint8_t*>(offs + 2 * ostride);
    const int xrow = nk * kBK / 2;                          // packed bytes per token in xs
    const uint32_t idesc = umma_idesc_f16(kBM, BN);
    const bool early = (p.flags & US_BITMAP_STATIC) != 0;   // weights may be fetched before the wait

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            us::mbar_init(&S.chunk_full[b], 1);
            us::mbar_init(&S.chunk_empty[b], kW4Dec);
        }
        for (int s = 0; s < kW4Stages; ++s) {
            us::mbar_init(&S.a_full[s], kW4Dec);
            us::mbar_init(&S.ab_empty[s], 1);
        }
        us::mbar_init(&S.x_full, 1);
        us::mbar_init(&S.done, 1);
        us::fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&S.tmem_base, 32);
    __syncthreads();
    tc_fence_after();
    us::pdl_launch_dependents();
    const uint32_t tmem = S.tmem_base;
    bool failed = false;
    int issued = 0;                                         // chunks issued (producer)

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (!early) us::pdl_wait();
        for (int i = lane; i <= nk; i += 32) {
            offs[i] = p.tile_off[(int64_t)(2 * mt) * p.nTK + kt0 + i];
            offs[ostride + i] = p.tile_off[(int64_t)(2 * mt + 1) * p.nTK + kt0 + i];
        }
        __syncwarp();
        // one chunk = up to kW4Chunk K steps of both bands: the tiles of a band's
        // K slice are consecutive, so four bulk copies move a whole chunk
        auto issue = [&](int c) {
            const int b = c & 1, q0 = c * kW4Chunk, ck = min(kW4Chunk, nk - q0);
            bool ok = true;
            if (lane < 2 * ck) {
                const int h = lane / ck, q = q0 + lane % ck;
                const uint32_t a = offs[h * ostride + q], e = offs[h * ostride + q + 1];
                ok = e >= a && (e - a) <= 4096u && (a & 31u) == 0 && (e & 31u) == 0 &&
                     (uint64_t)e * 4u <= p.values_bytes * 8ull;
            }
            const bool all_ok = __all_sync(0xffffffffu, ok);
            if (lane == 0) {
                if (!all_ok) us::set_status(p.status, US_ERR_CORRUPT);
                S.chunk_bad[b] = all_ok ? 0u : 1u;
                uint32_t vb[2];
                for (int h = 0; h < 2; ++h) vb[h] = all_ok ? (offs[h * ostride + q0 + ck] - offs[h * ostride + q0]) / 2u : 0u;
                uint8_t* dst = chunks + b * kW4ChunkBytes;
                us::mbar_arrive_expect_tx(&S.chunk_full[b], (uint32_t)(2 * ck * 512) + vb[0] + vb[1]);
                for (int h = 0; h < 2; ++h) {
                    const int64_t t = (int64_t)(2 * mt + h) * p.nTK + kt0 + q0;
                    us::bulk_g2s(dst + h * kW4BmBand, p.bitmap + t * 64, (uint32_t)(ck * 512), &S.chunk_full[b]);
                    if (vb[h])
                        us::bulk_g2s(dst + 2 * kW4BmBand + h * kW4ValBand, p.values + offs[h * ostride + q0] / 2u, vb[h],
                                     &S.chunk_full[b]);
                }
            }
            issued = c + 1;
        };
        int c = 0;
        if (early)
            for (; c < nchunks && c < 2; ++c) issue(c);
        us::pdl_wait();
        if (lane == 0) {
            us::mbar_arrive_expect_tx(&S.x_full, (uint32_t)(p.N * xrow));
            for (int n = 0; n < p.N; ++n)
                us::bulk_g2s(xs + n * xrow,
                             reinterpret_cast<const uint8_t*>(p.X) + ((int64_t)n * p.K + (int64_t)kt0 * kBK) / 2,
                             (uint32_t)xrow, &S.x_full);
        }
        for (; c < nchunks; ++c) {
            int stop = 0;
            if (c >= 2 && lane == 0 && !us::mbar_wait(&S.chunk_empty[c & 1], ((c >> 1) - 1) & 1, p.status)) stop = 1;
            if (__shfl_sync(0xffffffffu, stop, 0)) {
                failed = true;
                break;
            }
            issue(c);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            for (int q = 0; q < nk; ++q) {
                const int s = q % kW4Stages;
                if (!us::mbar_wait(&S.a_full[s], (q / kW4Stages) & 1, p.status)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = umma_smem_desc_sw128(a_st + s * kA);
                const uint64_t bd = umma_smem_desc_sw128(b_st + s * kB);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    umma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (q > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&S.ab_empty[s]);
            }
            umma_commit(&S.done);
        }
    } else {
        // ------------------------------------------------------------ decoders
        const int t = threadIdx.x - 64;                    // 0..255
        {
            const uint32_t sel = us::make_sel((uint32_t)t);
#pragma unroll
            for (int r = 0; r < kW4LutRep; ++r) lut[t * kW4LutRep + r] = sel;
            // absent tokens: zero activations (the bulk copies fill rows < N only)
            for (int i = t; i < (BN - p.N) * xrow / 4; i += 256)
                reinterpret_cast<uint32_t*>(xs + p.N * xrow)[i] = 0u;           // code 0 -> 0.0
        }
        us::named_bar_sync(1, 256);
        if (!us::mbar_wait(&S.x_full, 0, p.status)) failed = true;
        const int row = t >> 1, half = t & 1;
        const int band_h = row >> 6, i_in_band = row & 63;
        const uint32_t lut_lane = (uint32_t)(lane % kW4LutRep);
        for (int q = 0; q < nk && !failed; ++q) {
            const int c = q / kW4Chunk, b = c & 1, qq = q - c * kW4Chunk, s = q % kW4Stages;
            const int ck = min(kW4Chunk, nk - c * kW4Chunk);
            if (!us::mbar_wait(&S.chunk_full[b], (c >> 1) & 1, p.status)) {
                failed = true;
                break;
            }
            if (q >= kW4Stages && !us::mbar_wait(&S.ab_empty[s], ((q / kW4Stages) - 1) & 1, p.status)) {
                failed = true;
                break;
            }
            const uint8_t* buf = chunks + b * kW4ChunkBytes;
            const uint64_t* bm = reinterpret_cast<const uint64_t*>(buf + band_h * kW4BmBand + qq * 512);
            const uint64_t w0 = bm[lane], w1 = bm[lane + 32];
            const uint32_t packed = (uint32_t)__popcll(w0) | ((uint32_t)__popcll(w1) << 16);
            uint32_t incl = packed;
#pragma unroll
            for (int dd = 1; dd < 32; dd <<= 1) {
                const uint32_t o = __shfl_up_sync(0xffffffffu, incl, dd);
                if (lane >= dd) incl += o;
            }
            const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
            const uint32_t exr = __shfl_sync(0xffffffffu, incl - packed, i_in_band & 31);
            const uint32_t rowbase = (i_in_band < 32) ? (exr & 0xFFFFu) : (tot & 0xFFFFu) + (exr >> 16);
            const uint32_t* bo = offs + band_h * ostride;
            const bool ok = S.chunk_bad[b] == 0 && (tot & 0xFFFFu) + (tot >> 16) <= bo[q + 1] - bo[q];
            if (!ok && lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
            const uint64_t word = bm[i_in_band];
            const uint32_t bits = ok ? (half ? (uint32_t)(word >> 32) : (uint32_t)word) : 0u;
            const uint32_t o = rowbase + (half ? (uint32_t)__popc((uint32_t)word) : 0u);
            const uint32_t* vw = reinterpret_cast<const uint32_t*>(buf + 2 * kW4BmBand + band_h * kW4ValBand +
                                                                    (ok ? (bo[q] - bo[c * kW4Chunk]) / 2u : 0u));
            uint8_t* arow = a_st + s * kA + (row >> 3) * 1024 + (row & 7) * 128;
            // four independent byte-steps: each finds its own place in the run
            // (row base + popcount of the lower bits), so all are in flight at once
#pragma unroll
            for (int bt = 0; bt < 4; ++bt) {
                const uint32_t bb = (bits >> (8 * bt)) & 0xFFu;
                const uint32_t ob = o + (bt ? (uint32_t)__popc(bits & ((1u << (8 * bt)) - 1u)) : 0u);
                const uint32_t sel = lut[bb * kW4LutRep + lut_lane];
                const uint32_t c4 = (uint32_t)__popc(bb) << 2;
                const uint32_t wi = ob >> 3;
                const uint32_t nm = __funnelshift_r(vw[wi], vw[wi + 1], ob << 2) & ~us::shl_clamp(0xFFFFFFFFu, c4);
                const uint32_t even = (nm & 0x0F0F0F0Fu) ^ 0x08080808u;          // w + 8, ranks 0,2,4,6
                const uint32_t odd = ((nm >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;   // w + 8, ranks 1,3,5,7
                const int chunk = 4 * half + bt;
                *reinterpret_cast<uint4*>(arow + ((chunk ^ (row & 7)) << 4)) = i4x8_to_f16x8(even, odd, sel);
            }
            // activations of this K step: token n, 8 positions per thread
            if (t < BN * 8) {
                const int n = t >> 3, bt = t & 7;
                const uint32_t v = *reinterpret_cast<const uint32_t*>(xs + n * xrow + q * 32 + 4 * bt);
                const uint32_t lo = (v & 0x0F0F0F0Fu) ^ 0x08080808u, hi = ((v >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
                // lo holds elements 0,2,4,6 and hi 1,3,5,7: the all-set selector pair puts
                // element p at position p
                uint8_t* brow = b_st + s * kB + (n >> 3) * 1024 + (n & 7) * 128;
                *reinterpret_cast<uint4*>(brow + ((bt ^ (n & 7)) << 4)) = i4x8_to_f16x8(lo, hi, 0x73625140u);
            }
            us::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                us::mbar_arrive(&S.a_full[s]);
                if (qq == ck - 1) us::mbar_arrive(&S.chunk_empty[b]);
            }
        }
    }

    // ---------------------------------------------------------------- epilogue
    __syncthreads();
    const bool any_failed = __syncthreads_or(failed);
    int* part = reinterpret_cast<int*>(a_st);                // BN x 128 int32 (A stages idle)
    if (any_failed && warp == 0 && lane == 0) {
        // let this CTA's copies still in flight land (bounded) before it exits
        us::mbar_wait(&S.x_full, 0, nullptr);
        for (int c = issued > 2 ? issued - 2 : 0; c < issued; ++c)
            us::mbar_wait(&S.chunk_full[c & 1], (c >> 1) & 1, nullptr);
    }
    if (warp >= 2 && warp < 6) {
        // the final commit also covers MMAs issued before a failure: wait for it (bounded)
        const bool ready = us::mbar_wait(&S.done, 0, any_failed ? nullptr : p.status) && !any_failed;
        tc_fence_after();
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        if (BN == 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16), v);
#pragma unroll
            for (int c = 0; c < 16; ++c) part[c * kBM + row] = ready ? __float2int_rn(v[c]) : 0;
        } else {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16), v);
#pragma unroll
            for (int c = 0; c < 32; ++c) part[c * kBM + row] = ready ? __float2int_rn(v[c]) : 0;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 32);
    us::pdl_wait();                                          // before this grid's first global write
    const int m0 = mt * kBM;
    auto store = [&](int idx, int a) {
        const int n = idx / kBM, r = idx - n * kBM;
        if (n >= p.N || any_failed) return;
        const int m = m0 + r;
        const int64_t o = (int64_t)n * p.M + m;
        p.Yacc[o] = a;
        if (p.Y) {
            const float tt = __fmul_rn(__int2float_rn(a), us::half_bits_to_float(p.s_w[m]));
            p.Y[o] = us::float_to_half_bits(__fmul_rn(tt, us::half_bits_to_float(p.s_x[n])));
        }
    };
    if (p.split > 1) {
        us::cluster_sync();
        const int rank = (int)us::cluster_ctarank();
        // rank r reduces elements [r*total/split, (r+1)*total/split): any split, no remainder lost
        const int i0 = rank * (BN * kBM) / p.split, i1 = (rank + 1) * (BN * kBM) / p.split;
        for (int i = i0 + threadIdx.x; i < i1; i += kW4Threads) {
            int a = 0;
            for (int rr = 0; rr < p.split; ++rr) a += us::ld_cluster_s32(us::cluster_map(part + i, (uint32_t)rr));
            store(i, a);
        }
        us::cluster_sync();
    } else {
        for (int i = threadIdx.x; i < BN * kBM; i += kW4Threads) store(i, part[i]);
    }
}

size_t w4_smem(int BN, int nk) {
    return 1024 + kW4Stages * (kBM * kBK * 2 + BN * kBK * 2) + 2 * kW4ChunkBytes + 256 * kW4LutRep * 4 +
           ((sizeof(W4Smem) + 127) & ~size_t(127)) + (size_t)2 * ((nk + 1 + 3) & ~3) * 4 + (size_t)BN * nk * kBK / 2;
}

template <int BN>
us_status launch_w4(const UsKParams& p, cudaStream_t st) {
    const int nk = (p.nTK + p.split - 1) / p.split;
    const size_t smem = w4_smem(BN, nk);
    if (smem > 220 * 1024) return US_ERR_UNSUPPORTED;
    auto kern = w4a4_tc_kernel<BN>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return US_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.M / kBM) * p.split));
    cfg.blockDim = dim3(kW4Threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)p.split;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? US_OK : US_ERR_CUDA;
}

constexpr size_t kSmemBytes = 1024 + kStages * (kABytes + kBBytes) + kRawStages * kRawBytes + 256;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace

namespace us {

bool tc_f16_supported(int TM, int TK, int M, int N) {
    return TM == 64 && TK == 64 && M % kBM == 0 && N >= 64;
}

int tc_tok_block() { return kBN; }

int tc_split(int M, int N, int nTK) {
    const int ctas = (M / kBM) * ((N + kBN - 1) / kBN);
    int s = 1;
    while (ctas * s * 2 <= num_sms() && nTK / (s * 2) >= 8 && s < 8) s *= 2;
    return s;
}

size_t tc_ws(int M, int N, int split) {
    const int n_tiles = (N + kBN - 1) / kBN;
    const size_t counters = ((size_t)(M / kBM) * n_tiles * 4 + 255) & ~(size_t)255;
    return split <= 1 ? counters : counters + (size_t)split * n_tiles * M * kBN * 4;
}

bool tc_w4a4_supported(int TM, int TK, int M, int K, int N) {
    return TM == 64 && TK == 64 && M % kBM == 0 && K % 64 == 0 && N >= 8 && N <= 32;
}

int tc_w4a4_split(int M, int N, int nTK) {
    const int ctas = M / kBM;
    const int BN = N <= 16 ? 16 : 32;
    const int nk_max = 16 * 1024 / (BN * 32);            // packed activations of a CTA within 16 KB
    // two CTAs fit an SM: the largest cluster that still fills one wave, keeping
    // >= 4 K steps per slice; then grow further only if the activations do not fit
    int s = 1;
    while (s < 8 && ctas * s * 2 <= 2 * num_sms() && nTK / (s * 2) >= 4) s *= 2;
    while (s < 8 && (nTK + s - 1) / s > nk_max) s *= 2;
    return s;
}

bool tc_w4a4_fits(int N, int nTK, int split) {
    return w4_smem(N <= 16 ? 16 : 32, (nTK + split - 1) / split) <= 220 * 1024;
}

us_status launch_tc_w4a4(const UsKParams& p, cudaStream_t st) {
    return p.N <= 16 ? launch_w4<16>(p, st) : launch_w4<32>(p, st);
}

us_status launch_tc_f16(const UsKParams& p, cudaStream_t st) {
    auto enc = encode_fn();
    if (!enc) return US_ERR_CUDA;
    CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)p.K, (cuuint64_t)p.N};
    const cuuint64_t gstride[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBN};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(p.X), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return US_ERR_CUDA;
    TcParams tp;
    tp.p = p;
    tp.n_tiles = (p.N + kBN - 1) / kBN;
    if (cudaFuncSetAttribute(spmm_f16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
        cudaSuccess)
        return US_ERR_CUDA;
    dim3 grid((unsigned)(p.M / kBM), (unsigned)(tp.n_tiles * p.split));
    spmm_f16_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(tp, map);
    return cudaGetLastError() == cudaSuccess ? US_OK : US_ERR_CUDA;
}

}  // namespace us
