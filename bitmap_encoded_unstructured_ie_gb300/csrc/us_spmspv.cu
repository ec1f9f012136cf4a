// us_spmspv.cu -- fp16 spMspV with activation-skipped columns.
//
// y = (W (.) M) . (x (.) M(x)): static bitmap sparsity of W and a dynamic
// mask that keeps column k iff |x_k| > tau ("Unified Static-Dynamic Pruning
// for Efficient LLM Inference", section 2 and section 4.2, HAD-SMBD: an
// inactive column is skipped entirely; an active column's nonzeros are
// addressed by base + masked popcount).  W is stored column-major inside its
// tiles (Tiled-CBC scan, same page section 4.1), so the nonzeros of one
// column are one contiguous run: a skipped column costs no value bytes.
//
// Per CTA: one tile-row band x one K slice.  The tile bitmaps stream through
// a two-stage shared-memory ring (1-D bulk copies on mbarriers); the column
// bases come from a block scan of the column popcounts; each warp walks its
// columns, skips the inactive ones, and its lanes gather the active runs
// straight from global memory (read-once, no L1 allocation) into fp32 row
// accumulators.  Warp partials are summed in fixed warp order; split-K
// partials in fixed slice order by the last CTA of a band.
#include "us_common.cuh"
#include "us_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }

__device__ __forceinline__ uint16_t ld_stream_u16(const uint16_t* p) {
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

template <int TM>
__global__ void __launch_bounds__(kThreads)
spmspv_kernel(const UsKParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int WPC = TM / 64;          // 64-bit words per column
    constexpr int RPL = TM / 32;          // rows per lane
    const int TK = p.TK;
    const int band = blockIdx.x % p.nTM;
    const int slice = blockIdx.x / p.nTM;
    const int kt0 = (int)((int64_t)slice * p.nTK / p.split);
    const int kt1 = (int)((int64_t)(slice + 1) * p.nTK / p.split);
    const int nk = kt1 - kt0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    uint32_t off = 16;
    uint32_t* offs = reinterpret_cast<uint32_t*>(smem + off);
    off = align16(off + (uint32_t)(nk + 1) * 4u);
    const uint32_t bm_bytes = (uint32_t)TM * TK / 8u;
    uint8_t* stage_ptr[2];
    stage_ptr[0] = smem + off; off += align16(bm_bytes);
    stage_ptr[1] = smem + off; off += align16(bm_bytes);
    uint32_t* colbase = reinterpret_cast<uint32_t*>(smem + off); off = align16(off + (uint32_t)TK * 4u);
    float* xv = reinterpret_cast<float*>(smem + off); off = align16(off + (uint32_t)TK * 4u);
    float* red = reinterpret_cast<float*>(smem + off);      // kWarps x TM
    __shared__ uint32_t warp_tot[kWarps];
    __shared__ uint32_t tile_bad;
    __shared__ int flag_s;

    const int64_t tile0 = (int64_t)band * p.nTK + kt0;
    for (int q = threadIdx.x; q <= nk; q += kThreads) offs[q] = p.tile_off[tile0 + q];
    if (threadIdx.x == 0) {
        us::mbar_init(&bar[0], 1);
        us::mbar_init(&bar[1], 1);
        us::fence_mbar_init();
    }
    __syncthreads();
    const int nw = TM * TK / 64;
    auto issue = [&](int q) {
        const int s = q & 1;
        us::mbar_arrive_expect_tx(&bar[s], bm_bytes);
        us::bulk_g2s(stage_ptr[s], p.bitmap + (tile0 + q) * nw, bm_bytes, &bar[s]);
    };
    if (threadIdx.x == 0) {
        if (nk > 0) issue(0);
        if (nk > 1) issue(1);
    }

    float acc[RPL];
#pragma unroll
    for (int r = 0; r < RPL; ++r) acc[r] = 0.f;
    const uint16_t* vals16 = reinterpret_cast<const uint16_t*>(p.values);
    const uint16_t* x16 = reinterpret_cast<const uint16_t*>(p.X);

    uint32_t phase = 0;
    for (int q = 0; q < nk; ++q) {
        const int s = q & 1;
        const bool ok = us::mbar_wait(&bar[s], (phase >> s) & 1u, p.status);
        phase ^= 1u << s;
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) us::mbar_wait(&bar[s ^ 1], (phase >> (s ^ 1)) & 1u, nullptr);
            return;
        }
        const uint64_t* words = reinterpret_cast<const uint64_t*>(stage_ptr[s]);
        const int kbase = (kt0 + q) * TK;
        // column popcounts -> column bases; activation test
        uint32_t c = 0;
        if (threadIdx.x < TK) {
#pragma unroll
            for (int w = 0; w < WPC; ++w) c += (uint32_t)__popcll(words[threadIdx.x * WPC + w]);
            const float x = us::half_bits_to_float(x16[kbase + threadIdx.x]);
            xv[threadIdx.x] = (fabsf(x) > p.tau) ? x : 0.f;
        }
        {
            uint32_t incl = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += o;
            }
            if (lane == 31) warp_tot[warp] = incl;
            __syncthreads();
            uint32_t before = 0, P = 0;
#pragma unroll
            for (int i = 0; i < kWarps; ++i) {
                if (i < warp) before += warp_tot[i];
                P += warp_tot[i];
            }
            if (threadIdx.x < TK) colbase[threadIdx.x] = before + incl - c;
            if (threadIdx.x == 0) {
                const uint32_t o0 = offs[q], o1 = offs[q + 1];
                const bool good = o1 >= o0 && P <= o1 - o0 && (uint64_t)o1 * 2u <= p.values_bytes;
                tile_bad = good ? 0u : 1u;
                if (!good) us::set_status(p.status, US_ERR_CORRUPT);
            }
        }
        __syncthreads();
        if (!tile_bad) {
            const uint16_t* run = vals16 + offs[q];
            for (int j = warp; j < TK; j += kWarps) {
                const float xj = xv[j];
                if (xj == 0.f) continue;          // inactive (or zero) column: no value bytes read
                uint32_t base = colbase[j];
#pragma unroll
                for (int w = 0; w < WPC; ++w) {
                    const uint64_t word = words[j * WPC + w];
                    const uint32_t lo = (uint32_t)word, hi = (uint32_t)(word >> 32);
                    const uint32_t below = (1u << lane) - 1u;
                    if ((lo >> lane) & 1u) {
                        const uint32_t r = base + __popc(lo & below);
                        acc[2 * w] = fmaf(us::half_bits_to_float(ld_stream_u16(run + r)), xj, acc[2 * w]);
                    }
                    if ((hi >> lane) & 1u) {
                        const uint32_t r = base + __popc(lo) + __popc(hi & below);
                        acc[2 * w + 1] = fmaf(us::half_bits_to_float(ld_stream_u16(run + r)), xj, acc[2 * w + 1]);
                    }
                    base += __popc(lo) + __popc(hi);
                }
            }
        }
        __syncthreads();
        if (threadIdx.x == 0 && q + 2 < nk) issue(q + 2);
    }

    // rows: lane l of word w holds row 64w + l (acc[2w]) and 64w + 32 + l (acc[2w+1])
#pragma unroll
    for (int w = 0; w < WPC; ++w) {
        red[warp * TM + 64 * w + lane] = acc[2 * w];
        red[warp * TM + 64 * w + 32 + lane] = acc[2 * w + 1];
    }
    __syncthreads();
    float* part = reinterpret_cast<float*>(p.ws);
    for (int i = threadIdx.x; i < TM; i += kThreads) {
        float s = 0.f;
        for (int w = 0; w < kWarps; ++w) s += red[w * TM + i];
        if (p.split > 1) part[((int64_t)slice * p.nTM + band) * TM + i] = s;
        else p.Y[(int64_t)band * TM + i] = us::float_to_half_bits(s);
    }
    if (p.split <= 1) return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) flag_s = (atomicAdd(&p.counters[band], 1u) == (unsigned)p.split - 1u);
    __syncthreads();
    if (!flag_s) return;
    __threadfence();
    for (int i = threadIdx.x; i < TM; i += kThreads) {
        float s = 0.f;
        for (int sl = 0; sl < p.split; ++sl) {
            float* src = part + ((int64_t)sl * p.nTM + band) * TM + i;
            s += __ldcg(src);
            __stcg(src, 0.f);                   // leave the workspace zeroed for the next call
        }
        p.Y[(int64_t)band * TM + i] = us::float_to_half_bits(s);
    }
    if (threadIdx.x == 0) p.counters[band] = 0u;
}

size_t spmspv_smem(int TM, int TK, int nk) {
    auto a16 = [](size_t x) { return (x + 15) & ~(size_t)15; };
    size_t off = 16;
    off = a16(off + (size_t)(nk + 1) * 4);
    off += 2 * a16((size_t)TM * TK / 8);
    off = a16(off + (size_t)TK * 4);
    off = a16(off + (size_t)TK * 4);
    off += (size_t)kWarps * TM * 4;
    return off;
}

template <int TM>
us_status launch_t(const UsKParams& p, cudaStream_t st) {
    const int nk = (p.nTK + p.split - 1) / p.split;
    const size_t smem = spmspv_smem(TM, p.TK, nk);
    if (smem > 227 * 1024) return US_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(spmspv_kernel<TM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return US_ERR_CUDA;
    spmspv_kernel<TM><<<(unsigned)(p.nTM * p.split), kThreads, smem, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? US_OK : US_ERR_CUDA;
}

}  // namespace

namespace us {

size_t spmspv_ws(int M, int TM, int split) {
    const int nTM = M / TM;
    const size_t counters = ((size_t)nTM * 4 + 255) & ~(size_t)255;
    return split <= 1 ? counters : counters + (size_t)split * M * 4;
}

us_status launch_spmspv(const UsKParams& p, cudaStream_t st) {
    switch (p.TM) {
        case 64: return launch_t<64>(p, st);
        case 128: return launch_t<128>(p, st);
        case 256: return launch_t<256>(p, st);
    }
    return US_ERR_UNSUPPORTED;
}

}  // namespace us
