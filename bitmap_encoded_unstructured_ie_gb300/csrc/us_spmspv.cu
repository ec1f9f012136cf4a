// us_spmspv.cu -- fp16 spMspV with activation-skipped columns.
//
// y = (W (.) M) . (x (.) M(x)): static bitmap sparsity of W and a dynamic
// mask that keeps column k iff |x_k| > tau ("Unified Static-Dynamic Pruning
// for Efficient LLM Inference", section 2 and section 4.2: an inactive column
// is skipped entirely; an active column's nonzeros are addressed by its base
// plus a masked popcount, HAD-SMBD).  W is stored column-major inside its
// tiles (Tiled-CBC scan, same page section 4.1), so the nonzeros of one
// column form one contiguous run: a skipped column costs no value bytes.
//
// Per CTA: one tile-row band x one K slice; the K slices of a band form one
// thread-block cluster.  Eight warps, each owning whole tiles, with no block
// barrier in the main loop:
//  * a warp fetches its next tile's bitmap (16 bytes per lane, read-only
//    path) while it works on the current one - the metadata-first prefetch of
//    SPDP section 4.2.2;
//  * column popcounts -> column bases by warp scan; a ballot of
//    "popcount > 0 and |x_j| > tau" lists the active columns;
//  * for each active column the lanes own rows: a set bit yields
//    rank = base + masked popcount, and the value run[rank] is gathered
//    straight from global memory (one column's run is contiguous, so a warp's
//    loads coalesce); four columns' loads are issued before they are used;
//  * fp32 row accumulators; warp partials are summed in fixed warp order and
//    the slices of a band in fixed rank order through distributed shared
//    memory (no workspace, bitwise reproducible).
#include "us_common.cuh"
#include "us_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
#ifndef US_SPMSPV_BATCH
#define US_SPMSPV_BATCH 8            // measured on 14336 x 4096: 4 -> 64 / 25 us, 8 -> 53 / 22 us (50 / 90 % zeros)
#endif
constexpr int kBatch = US_SPMSPV_BATCH;   // active columns whose loads are in flight together

__device__ __forceinline__ uint16_t ld_once_u16(const uint16_t* p) {
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_once_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// TM rows per tile; NPV 16-byte pieces of a tile's bitmap held per lane
template <int TM, int NPV>
__global__ void __launch_bounds__(kThreads)
spmspv_kernel(const UsKParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int WPC = TM / 64;          // 64-bit words per column
    constexpr int RPL = TM / 32;          // rows per lane
    const int TK = p.TK;
    const int band = blockIdx.x / p.split;        // the split slices of a band form one cluster
    const int slice = blockIdx.x % p.split;
    const int kt0 = (int)((int64_t)slice * p.nTK / p.split);
    const int kt1 = (int)((int64_t)(slice + 1) * p.nTK / p.split);
    const int nk = kt1 - kt0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bm_bytes = (uint32_t)TM * TK / 8u;            // <= NPV * 512 (launcher checks)
    const uint32_t bm_vec = bm_bytes / 16u;                       // 16-byte pieces
    const int nw = TM * TK / 64;

    // shared memory: per-warp bitmap and column-base scratch, activations, reduction
    uint64_t* wbm = reinterpret_cast<uint64_t*>(smem) + (size_t)warp * (bm_bytes / 8u);
    uint32_t off = kWarps * bm_bytes;
    uint32_t* wbase = reinterpret_cast<uint32_t*>(smem + off) + warp * TK;
    off += kWarps * TK * 4;
    // sized for the longest slice so that every CTA of the cluster has the same
    // layout: the reduction reads the other CTAs' partials at this CTA's offset
    const int nk_max = (p.nTK + p.split - 1) / p.split;
    float* xs = reinterpret_cast<float*>(smem + off);             // nk x TK (masked activations)
    off += ((uint32_t)nk_max * TK * 4u + 15u) & ~15u;
    float* red = reinterpret_cast<float*>(smem + off);            // kWarps x TM, then TM

    us::pdl_launch_dependents();
    us::pdl_wait();
    {
        const uint16_t* x16 = reinterpret_cast<const uint16_t*>(p.X) + (int64_t)kt0 * TK;
        for (int i = threadIdx.x; i < nk * TK; i += kThreads) {
            const float x = us::half_bits_to_float(x16[i]);
            xs[i] = (fabsf(x) > p.tau) ? x : 0.f;                     // the dynamic mask M(x)
        }
    }
    __syncthreads();

    float acc[RPL];
#pragma unroll
    for (int r = 0; r < RPL; ++r) acc[r] = 0.f;
    const uint16_t* vals16 = reinterpret_cast<const uint16_t*>(p.values);
    const int64_t tile0 = (int64_t)band * p.nTK + kt0;

    // prefetch registers for the next tile of this warp
    uint4 nbm[NPV];
#pragma unroll
    for (int v = 0; v < NPV; ++v) nbm[v] = make_uint4(0, 0, 0, 0);
    uint32_t no0 = 0, no1 = 0;
    auto fetch = [&](int q) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.bitmap + (tile0 + q) * nw);
#pragma unroll
        for (int v = 0; v < NPV; ++v) {
            const uint32_t piece = (uint32_t)lane + 32u * v;
            if (piece < bm_vec) nbm[v] = ld_once_v4(src + 16u * piece);
        }
        no0 = __ldg(p.tile_off + tile0 + q);
        no1 = __ldg(p.tile_off + tile0 + q + 1);
    };
    if (warp < nk) fetch(warp);

    for (int q = warp; q < nk; q += kWarps) {
        // ---- this tile's bitmap into the warp's scratch; next tile's in flight
#pragma unroll
        for (int v = 0; v < NPV; ++v) {
            const uint32_t piece = (uint32_t)lane + 32u * v;
            if (piece < bm_vec) reinterpret_cast<uint4*>(wbm)[piece] = nbm[v];
        }
        const uint32_t o0 = no0, o1 = no1;
        if (q + kWarps < nk) fetch(q + kWarps);
        __syncwarp();
        // ---- column popcounts -> bases (warp scan); active columns
        uint32_t run_sum = 0;                            // columns of the earlier 32-column groups
        uint32_t actmask[4] = {0u, 0u, 0u, 0u};          // up to 128 columns
        const float* xq = xs + q * TK;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if (g * 32 >= TK) break;
            const int j = g * 32 + lane;
            uint32_t c = 0;
            bool act = false;
            if (j < TK) {
#pragma unroll
                for (int w = 0; w < WPC; ++w) c += (uint32_t)__popcll(wbm[j * WPC + w]);
                act = c > 0 && xq[j] != 0.f;
            }
            uint32_t incl = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += o;
            }
            if (j < TK) wbase[j] = run_sum + incl - c;
            run_sum += __shfl_sync(0xffffffffu, incl, 31);
            actmask[g] = __ballot_sync(0xffffffffu, act);
        }
        const uint32_t P = run_sum;
        const bool good = o1 >= o0 && (o1 - o0) <= (uint32_t)(TM * TK) && (uint64_t)o1 * 2u <= p.values_bytes &&
                          P <= o1 - o0;
        if (!good) {
            if (lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
            __syncwarp();
            continue;
        }
        __syncwarp();
        const uint16_t* run = vals16 + o0;
        const uint32_t below = (1u << lane) - 1u;
        // ---- active columns, kBatch at a time: issue every gather, then use them
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            uint32_t m = actmask[g];
            while (m) {
                int js[kBatch];
#pragma unroll
                for (int t = 0; t < kBatch; ++t) {
                    js[t] = -1;
                    if (m) {
                        js[t] = g * 32 + __ffs(m) - 1;
                        m &= m - 1;
                    }
                }
                uint16_t v[kBatch][2 * WPC];
                float xj[kBatch];
#pragma unroll
                for (int t = 0; t < kBatch; ++t) {
                    const int j = js[t];
                    xj[t] = 0.f;
#pragma unroll
                    for (int h = 0; h < 2 * WPC; ++h) v[t][h] = 0;
                    if (j < 0) continue;
                    xj[t] = xq[j];
                    uint32_t base = wbase[j];
#pragma unroll
                    for (int w = 0; w < WPC; ++w) {
                        const uint64_t word = wbm[j * WPC + w];
                        const uint32_t lo = (uint32_t)word, hi = (uint32_t)(word >> 32);
                        if ((lo >> lane) & 1u) v[t][2 * w] = ld_once_u16(run + base + __popc(lo & below));
                        if ((hi >> lane) & 1u)
                            v[t][2 * w + 1] = ld_once_u16(run + base + __popc(lo) + __popc(hi & below));
                        base += __popc(lo) + __popc(hi);
                    }
                }
#pragma unroll
                for (int t = 0; t < kBatch; ++t)
#pragma unroll
                    for (int h = 0; h < 2 * WPC; ++h)
                        acc[h] = fmaf(us::half_bits_to_float(v[t][h]), xj[t], acc[h]);
            }
        }
        __syncwarp();
    }

    // ---- rows: lane l of word w holds row 64w + l (acc[2w]) and 64w + 32 + l (acc[2w+1])
    __syncthreads();
#pragma unroll
    for (int w = 0; w < WPC; ++w) {
        red[warp * TM + 64 * w + lane] = acc[2 * w];
        red[warp * TM + 64 * w + 32 + lane] = acc[2 * w + 1];
    }
    __syncthreads();
    float* outv = red + kWarps * TM;
    for (int i = threadIdx.x; i < TM; i += kThreads) {
        float s = 0.f;
        for (int w = 0; w < kWarps; ++w) s += red[w * TM + i];
        outv[i] = s;
    }
    __syncthreads();
    if (p.split > 1) {
        us::cluster_sync();
        const int rank = (int)us::cluster_ctarank();
        const int i0 = rank * TM / p.split, i1 = (rank + 1) * TM / p.split;
        for (int i = i0 + threadIdx.x; i < i1; i += kThreads) {
            float s = 0.f;
            for (int r = 0; r < p.split; ++r) s += us::ld_cluster_f32(us::cluster_map(outv + i, (uint32_t)r));
            p.Y[(int64_t)band * TM + i] = us::float_to_half_bits(s);
        }
        us::cluster_sync();
    } else {
        for (int i = threadIdx.x; i < TM; i += kThreads) p.Y[(int64_t)band * TM + i] = us::float_to_half_bits(outv[i]);
    }
}

size_t spmspv_smem(int TM, int TK, int nk) {
    size_t off = (size_t)kWarps * TM * TK / 8;
    off += (size_t)kWarps * TK * 4;
    off += ((size_t)nk * TK * 4 + 15) & ~(size_t)15;
    off += (size_t)(kWarps + 1) * TM * 4;
    return off;
}

template <int TM, int NPV>
us_status launch_t(const UsKParams& p, cudaStream_t st) {
    const int nk = (p.nTK + p.split - 1) / p.split;
    const size_t smem = spmspv_smem(TM, p.TK, nk);
    if (smem > 220 * 1024) return US_ERR_UNSUPPORTED;
    auto kern = spmspv_kernel<TM, NPV>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return US_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.nTM * p.split));
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
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? US_OK : US_ERR_CUDA;
}

}  // namespace

namespace us {

size_t spmspv_ws(int, int, int) { return 0; }     // slices reduce inside the cluster

int spmspv_max_split() { return 8; }

template <int TM>
us_status launch_tm(const UsKParams& p, cudaStream_t st) {
    const int bm_bytes = TM * p.TK / 8;                  // 128 .. 4096
    if (bm_bytes <= 512) return launch_t<TM, 1>(p, st);
    if (bm_bytes <= 1024) return launch_t<TM, 2>(p, st);
    if (bm_bytes <= 2048) return launch_t<TM, 4>(p, st);
    return launch_t<TM, 8>(p, st);
}

us_status launch_spmspv(const UsKParams& p, cudaStream_t st) {
    switch (p.TM) {
        case 64: return launch_tm<64>(p, st);
        case 128: return launch_tm<128>(p, st);
        case 256: return launch_tm<256>(p, st);
    }
    return US_ERR_UNSUPPORTED;
}

}  // namespace us
