// us_spmspv_ci.cu -- ColInfo and the batched fp16 spMspV that reads it.
//
// ColInfo ("Unified Static-Dynamic Pruning for Efficient LLM Inference",
// section 4.1, Tiled-CBC storage structure): for a COL-order matrix, one
// 32-bit word per column of every tile, tile-major; upper 16 bits the column's
// starting offset inside the tile's value run, lower 16 bits its nonzero count.
// With it a kernel finds an active column's values without reading the bitmap
// words of the columns before it, so an inactive column costs 4 bytes of
// metadata instead of TM / 8 bytes of bitmap (SPDP section 4.2: the column
// metadata is fetched first, then only the activation-relevant data).
//
// Batched dynamic pruning: token n keeps X[n][k] iff |X[n][k]| > tau; a
// column is fetched iff it is active for some token of the CTA's token block.
//
// Per CTA: one tile-row band x one K slice x one block of NB tokens; the K
// slices of a band form one thread-block cluster and reduce through
// distributed shared memory in fixed rank order.  Eight warps own whole tiles:
//  * the ColInfo of the warp's tile two ahead is fetched while a warp ballot
//    lists the active columns of the next tile and each lane sends for one of
//    their bitmap words (metadata first, data second);
//  * for each column the lanes own rows: a set bit gives rank = offset +
//    masked popcount, and run[rank] is gathered (one column's run is
//    contiguous, so a warp's loads coalesce);
//  * fp32 accumulators per row and token; warp partials summed in fixed order.
#include "us_common.cuh"
#include "us_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxTK = 128;

__device__ __forceinline__ uint16_t ld_once_u16(const uint16_t* p) {
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// ------------------------------------------------------------------ ColInfo
// One warp per tile: lane l counts columns l, l + 32, ...; a warp scan over
// the column counts gives the offsets.
template <int TM>
__global__ void __launch_bounds__(kThreads) colinfo_kernel(const uint64_t* __restrict__ bitmap, int TK, int64_t nT,
                                                           uint32_t* __restrict__ colinfo) {
    constexpr int WPC = TM / 64;
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= nT) return;
    const uint64_t* bm = bitmap + t * (int64_t)(TM / 64) * TK;
    uint32_t run = 0;
    for (int g = 0; g * 32 < TK; ++g) {
        const int j = g * 32 + lane;
        uint32_t c = 0;
        if (j < TK) {
#pragma unroll
            for (int w = 0; w < WPC; ++w) c += (uint32_t)__popcll(__ldg(bm + (int64_t)j * WPC + w));
        }
        uint32_t incl = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += o;
        }
        if (j < TK) colinfo[t * TK + j] = ((run + incl - c) << 16) | c;
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
}

// ------------------------------------------------------------------ spMspV
// TM rows per tile, NB tokens per CTA
template <int TM, int NB>
__global__ void __launch_bounds__(kThreads, TM >= 128 ? 2 : 3)   // 64-row tiles: three per SM, so the usual
                                                                    // grid of bands x 2 K slices is one wave
spmspv_ci_kernel(const UsKParams p, const uint32_t* __restrict__ colinfo) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int WPC = TM / 64;            // 64-bit words per column
    constexpr int RPL = TM / 32;            // rows per lane
    constexpr int kB = 8 / WPC;             // active columns whose values are in flight together
    const int TK = p.TK;
    const int band = blockIdx.x / p.split;
    const int slice = blockIdx.x % p.split;
    const int n0 = blockIdx.y * NB;
    const int nb = min(NB, p.N - n0);
    const int kt0 = (int)((int64_t)slice * p.nTK / p.split);
    const int kt1 = (int)((int64_t)(slice + 1) * p.nTK / p.split);
    const int nk = kt1 - kt0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = TM * TK / 64;            // bitmap words per tile
    const int cpl = (TK + 31) / 32;         // ColInfo words per lane

    // shared memory (the same layout in every CTA of the cluster: the reduction
    // reads the other CTAs' sums at this CTA's offset, so it is sized for the
    // longest slice): masked activations NB x nk_max x TK, union-active bits,
    // per-warp active-column lists, reduction
    const int nk_max = (p.nTK + p.split - 1) / p.split;
    const int npos = nk_max * TK;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                  // fp16: an fp16 input stays exact
    uint32_t* actw = reinterpret_cast<uint32_t*>(smem + (((size_t)NB * npos * 2 + 15) & ~(size_t)15));
    uint32_t* lists = actw + (npos + 31) / 32;                       // kWarps x 2 x TK x {j, ColInfo}
    uint32_t* mylist = lists + warp * 2 * TK * 2;
    uint32_t* wlists = lists + kWarps * 2 * TK * 2;                  // kWarps x TK x WPC words
    float* red = reinterpret_cast<float*>(wlists + kWarps * TK * WPC * 2);   // kWarps x NB x TM, then NB x TM

    us::pdl_launch_dependents();
    us::pdl_wait();
    {
        // masked activations and, per position, "active for some token"
        const uint16_t* x16 = reinterpret_cast<const uint16_t*>(p.X);
        const int total = nk * TK;
        for (int i0 = warp * 32; i0 < ((total + 31) & ~31); i0 += kThreads) {
            const int i = i0 + lane;
            bool any = false;
            for (int n = 0; n < NB; ++n) {
                uint16_t xm = 0;
                if (i < total && n < nb) {
                    const uint16_t xb = x16[(int64_t)(n0 + n) * p.K + (int64_t)kt0 * TK + i];
                    if (fabsf(us::half_bits_to_float(xb)) > p.tau) xm = xb;   // the dynamic mask M(x)
                }
                if (i < total) xs[n * npos + i] = xm;
                any |= (xm & 0x7FFFu) != 0;
            }
            const uint32_t m = __ballot_sync(0xffffffffu, any);
            if (lane == 0) actw[i0 / 32] = m;
        }
    }
    __syncthreads();

    float acc[NB][RPL];
#pragma unroll
    for (int n = 0; n < NB; ++n)
#pragma unroll
        for (int r = 0; r < RPL; ++r) acc[n][r] = 0.f;
    const uint16_t* vals16 = reinterpret_cast<const uint16_t*>(p.values);
    const int64_t tile0 = (int64_t)band * p.nTK + kt0;
    const uint32_t below = (1u << lane) - 1u;

    // A three-stage pipeline per warp (SPDP section 4.2.2: metadata first,
    // data second): the ColInfo of the tile two ahead is in flight, the bitmap
    // words of the next tile's active columns are in flight (lane e fetches
    // list entry e), and the current tile's values are gathered.
    uint32_t* wl = wlists + (size_t)warp * TK * WPC * 2;          // current tile's words (as 2 x 32 bits)
    auto load_ci = [&](int q, uint32_t (&c)[kMaxTK / 32]) {
#pragma unroll
        for (int k = 0; k < kMaxTK / 32; ++k) {
            const int j = k * 32 + lane;
            c[k] = (q < nk && k < cpl && j < TK) ? __ldg(colinfo + (tile0 + q) * TK + j) : 0u;
        }
    };
    // the active columns of tile q into list `buf` (j and ColInfo per entry);
    // returns their number, or -1 when the ColInfo overruns the tile's run
    auto build_list = [&](int q, const uint32_t (&c)[kMaxTK / 32], uint32_t len, uint32_t* buf) -> int {
        int nact = 0;
        bool ok = true;
#pragma unroll
        for (int k = 0; k < kMaxTK / 32; ++k) {
            if (k >= cpl) break;
            const int j = k * 32 + lane;
            const int pos = q * TK + j;
            const uint32_t nnz = c[k] & 0xFFFFu, off = c[k] >> 16;
            const bool in = j < TK;
            ok &= !in || (nnz <= (uint32_t)TM && off + nnz <= len);
            const bool act = in && nnz > 0 && ((actw[pos >> 5] >> (pos & 31)) & 1u);
            const uint32_t m = __ballot_sync(0xffffffffu, act);
            if (act) {
                const int e = nact + __popc(m & below);
                buf[2 * e] = (uint32_t)j;
                buf[2 * e + 1] = c[k];
            }
            nact += __popc(m);
        }
        __syncwarp();
        return __all_sync(0xffffffffu, ok) ? nact : -1;
    };
    // lane e (and e + 32, ...) fetches the bitmap words of list entry e
    uint64_t wreg[kMaxTK / 32][WPC];
    auto load_words = [&](int q, const uint32_t* buf, int nact) {
        const uint64_t* tbm = p.bitmap + (tile0 + q) * nw;
#pragma unroll
        for (int k = 0; k < kMaxTK / 32; ++k) {
            const int e = k * 32 + lane;
#pragma unroll
            for (int v = 0; v < WPC; ++v) wreg[k][v] = e < nact ? __ldg(tbm + (int64_t)buf[2 * e] * WPC + v) : 0ull;
        }
    };
    auto run_len = [&](int q, uint32_t& o0, uint32_t& len) -> bool {
        if (q >= nk) return false;
        o0 = __ldg(p.tile_off + tile0 + q);
        const uint32_t o1 = __ldg(p.tile_off + tile0 + q + 1);
        len = o1 - o0;
        return o1 >= o0 && len <= (uint32_t)(TM * TK) && (uint64_t)o1 * 2u <= p.values_bytes;
    };

    // prologue: tile q0 = warp listed and its words in flight, ColInfo of q0 + kWarps in flight
    int cur = 0;
    int nact_cur = 0;
    uint32_t o0_cur = 0, len_cur = 0;
    bool run_ok_cur = false;
    uint32_t ci_a[kMaxTK / 32];
    if (warp < nk) {
        uint32_t c0[kMaxTK / 32];
        load_ci(warp, c0);
        run_ok_cur = run_len(warp, o0_cur, len_cur);
        nact_cur = build_list(warp, c0, len_cur, mylist);
        load_words(warp, mylist, nact_cur);
        load_ci(warp + kWarps, ci_a);
    }

    for (int q = warp; q < nk; q += kWarps) {
        uint32_t* lcur = mylist + cur * TK * 2;
        uint32_t* lnxt = mylist + (cur ^ 1) * TK * 2;
        // (a) the current tile's words have landed: into the warp's word list
#pragma unroll
        for (int k = 0; k < kMaxTK / 32; ++k) {
            const int e = k * 32 + lane;
            if (e < nact_cur)
#pragma unroll
                for (int v = 0; v < WPC; ++v) {
                    wl[(e * WPC + v) * 2] = (uint32_t)wreg[k][v];
                    wl[(e * WPC + v) * 2 + 1] = (uint32_t)(wreg[k][v] >> 32);
                }
        }
        __syncwarp();
        // (b) the next tile: list it, send for its words; (c) ColInfo two ahead
        const int qn = q + kWarps;
        int nact_nxt = 0;
        uint32_t o0_nxt = 0, len_nxt = 0;
        bool run_ok_nxt = false;
        if (qn < nk) {
            run_ok_nxt = run_len(qn, o0_nxt, len_nxt);
            nact_nxt = build_list(qn, ci_a, len_nxt, lnxt);
            load_words(qn, lnxt, nact_nxt);
            load_ci(qn + kWarps, ci_a);
        }
        // (d) this tile's values, kB active columns per round trip
        if (nact_cur < 0 || !run_ok_cur) {
            if (lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
        } else {
            const uint16_t* run = vals16 + o0_cur;
            for (int e0 = 0; e0 < nact_cur; e0 += kB) {
                uint16_t v[kB][2 * WPC];
                int xpos[kB];
#pragma unroll
                for (int b = 0; b < kB; ++b) {
                    const int e = e0 + b;
#pragma unroll
                    for (int h = 0; h < 2 * WPC; ++h) v[b][h] = 0;
                    xpos[b] = -1;
                    if (e >= nact_cur) continue;
                    const int j = (int)lcur[2 * e];
                    const uint32_t cw = lcur[2 * e + 1];
                    const uint32_t lim = (cw >> 16) + (cw & 0xFFFFu);  // end of the column's values
                    uint32_t base = cw >> 16;
                    xpos[b] = q * TK + j;
#pragma unroll
                    for (int w = 0; w < WPC; ++w) {
                        const uint32_t lo = wl[(e * WPC + w) * 2], hi = wl[(e * WPC + w) * 2 + 1];
                        const uint32_t r0 = base + __popc(lo & below), r1 = base + __popc(lo) + __popc(hi & below);
                        // a rank past the column's count means bitmap and ColInfo disagree
                        if ((lo >> lane) & 1u) v[b][2 * w] = r0 < lim ? ld_once_u16(run + r0) : (uint16_t)0;
                        if ((hi >> lane) & 1u) v[b][2 * w + 1] = r1 < lim ? ld_once_u16(run + r1) : (uint16_t)0;
                        base += __popc(lo) + __popc(hi);
                    }
                    if (base != lim) us::set_status(p.status, US_ERR_CORRUPT);
                }
#pragma unroll
                for (int b = 0; b < kB; ++b) {
                    if (xpos[b] < 0) break;
#pragma unroll
                    for (int n = 0; n < NB; ++n) {
                        const float xj = us::half_bits_to_float(xs[n * npos + xpos[b]]);
#pragma unroll
                        for (int h = 0; h < 2 * WPC; ++h)
                            acc[n][h] = fmaf(us::half_bits_to_float(v[b][h]), xj, acc[n][h]);
                    }
                }
            }
        }
        __syncwarp();
        cur ^= 1;
        nact_cur = nact_nxt;
        o0_cur = o0_nxt;
        len_cur = len_nxt;
        run_ok_cur = run_ok_nxt;
    }

    // ---- rows: lane l of word w holds row 64w + l (acc[.][2w]) and 64w + 32 + l
    __syncthreads();
#pragma unroll
    for (int n = 0; n < NB; ++n)
#pragma unroll
        for (int w = 0; w < WPC; ++w) {
            red[(warp * NB + n) * TM + 64 * w + lane] = acc[n][2 * w];
            red[(warp * NB + n) * TM + 64 * w + 32 + lane] = acc[n][2 * w + 1];
        }
    __syncthreads();
    float* outv = red + kWarps * NB * TM;
    for (int i = threadIdx.x; i < NB * TM; i += kThreads) {
        const int n = i / TM, r = i - n * TM;
        float s = 0.f;
        for (int w = 0; w < kWarps; ++w) s += red[(w * NB + n) * TM + r];
        outv[i] = s;
    }
    __syncthreads();
    if (p.split > 1) {
        us::cluster_sync();
        const int rank = (int)us::cluster_ctarank();
        const int i0 = rank * NB * TM / p.split, i1 = (rank + 1) * NB * TM / p.split;
        for (int i = i0 + threadIdx.x; i < i1; i += kThreads) {
            const int n = i / TM, r = i - n * TM;
            float s = 0.f;
            for (int c = 0; c < p.split; ++c) s += us::ld_cluster_f32(us::cluster_map(outv + i, (uint32_t)c));
            if (n < nb) p.Y[(int64_t)(n0 + n) * p.M + (int64_t)band * TM + r] = us::float_to_half_bits(s);
        }
        us::cluster_sync();
    } else {
        for (int i = threadIdx.x; i < nb * TM; i += kThreads) {
            const int n = i / TM, r = i - n * TM;
            p.Y[(int64_t)(n0 + n) * p.M + (int64_t)band * TM + r] = us::float_to_half_bits(outv[i]);
        }
    }
}

size_t spmspv_ci_smem(int TM, int TK, int nk_max, int NB) {
    const size_t npos = (size_t)nk_max * TK;
    size_t b = ((size_t)NB * npos * 2 + 15) & ~(size_t)15;  // xs (fp16)
    b += (npos + 31) / 32 * 4;                              // active bits
    b += (size_t)kWarps * 2 * TK * 2 * 4;                   // active-column lists, two per warp
    b += (size_t)kWarps * TK * (TM / 64) * 8;               // their bitmap words
    b += (size_t)(kWarps + 1) * NB * TM * 4;                // reduction
    return b;
}

template <int TM, int NB>
us_status launch_ci_t(const UsKParams& p, const uint32_t* colinfo, cudaStream_t st) {
    const int nk_max = (p.nTK + p.split - 1) / p.split;
    const size_t smem = spmspv_ci_smem(TM, p.TK, nk_max, NB);
    if (smem > 220 * 1024) return US_ERR_UNSUPPORTED;
    auto kern = spmspv_ci_kernel<TM, NB>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return US_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.nTM * p.split), (unsigned)((p.N + NB - 1) / NB));
    cfg.blockDim = dim3(kThreads);
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
    return cudaLaunchKernelEx(&cfg, kern, p, colinfo) == cudaSuccess ? US_OK : US_ERR_CUDA;
}

// tokens per CTA: up to 8, with at most 16 accumulators per lane, and fewer
// when the staged activations would not fit in shared memory
template <int TM>
us_status launch_ci_tm(const UsKParams& p, const uint32_t* colinfo, cudaStream_t st) {
    constexpr int kMaxNB = 16 / (TM / 32);                  // 8, 4, 2
    const int nk_max = (p.nTK + p.split - 1) / p.split;
    int nb = p.N < kMaxNB ? p.N : kMaxNB;
    while (nb > 1 && spmspv_ci_smem(TM, p.TK, nk_max, nb) > 220 * 1024) nb /= 2;
    if (nb <= 1) return launch_ci_t<TM, 1>(p, colinfo, st);
    if (nb <= 2) return launch_ci_t<TM, 2>(p, colinfo, st);
    if constexpr (kMaxNB >= 4) {
        if (nb <= 4) return launch_ci_t<TM, 4>(p, colinfo, st);
    }
    if constexpr (kMaxNB >= 8) return launch_ci_t<TM, 8>(p, colinfo, st);
    return US_ERR_UNSUPPORTED;
}

}  // namespace

namespace us {

us_status launch_colinfo(const uint64_t* bitmap, int TM, int TK, int64_t nT, uint32_t* colinfo, cudaStream_t st) {
    if (nT <= 0) return US_OK;
    const dim3 grid((unsigned)((nT + kWarps - 1) / kWarps));
    switch (TM) {
        case 64: colinfo_kernel<64><<<grid, kThreads, 0, st>>>(bitmap, TK, nT, colinfo); break;
        case 128: colinfo_kernel<128><<<grid, kThreads, 0, st>>>(bitmap, TK, nT, colinfo); break;
        case 256: colinfo_kernel<256><<<grid, kThreads, 0, st>>>(bitmap, TK, nT, colinfo); break;
        default: return US_ERR_UNSUPPORTED;
    }
    return cudaGetLastError() == cudaSuccess ? US_OK : US_ERR_CUDA;
}

us_status launch_spmspv_ci(const UsKParams& p, const uint32_t* colinfo, cudaStream_t st) {
    if (p.TK > kMaxTK) return US_ERR_UNSUPPORTED;
    switch (p.TM) {
        case 64: return launch_ci_tm<64>(p, colinfo, st);
        case 128: return launch_ci_tm<128>(p, colinfo, st);
        case 256: return launch_ci_tm<256>(p, colinfo, st);
    }
    return US_ERR_UNSUPPORTED;
}

}  // namespace us
