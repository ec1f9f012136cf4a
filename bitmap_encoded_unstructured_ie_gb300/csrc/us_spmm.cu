// us_spmm.cu -- generic bitmap-tile SpMM on CUDA cores (any tile shape, any N).
//
// Y = W . X for W stored as bitmap tiles (IE-BME of "UnionSparse: An
// Index-Efficient Sparsity Framework for Low-Bit Sparse LLM Inference on
// Edge", section V-A, one area; row-major scan).  This is the general path:
// every supported tile shape, both element types, any token count.  The
// specialised kernels (W4A4 register decode, tensor-core prefill) take the
// common shapes; this one keeps every other shape on the GPU.
//
// Per CTA: one tile-row band (TM rows) x one K slice x one block of up to 32
// tokens.  The producer thread streams each K tile's bitmap words and value
// run into a two-stage shared-memory ring with 1-D bulk copies (TMA) that
// complete on mbarriers (the prefetch/compute overlap of UnionSparse's
// DW-PC pipeline, section VI-A).  All threads then
//   1. build the word prefix of popcounts (block scan),
//   2. decode every position: rank = word prefix + popcount of the lower
//      bits of its word, value = run[rank] or 0 (UnionSparse section VI-B,
//      rank addressing),
//   3. multiply the decoded tile by the staged activations.
// Split-K partials go to the workspace; the last CTA of a band reduces them
// in fixed slice order (deterministic) and applies the epilogue.
#include "us_common.cuh"
#include "us_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kTB = 32;                 // tokens per CTA

__device__ __forceinline__ uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }

// exclusive scan of (c0 + c1) over the block; returns the prefix, writes total
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) {
        const uint32_t s = warp_tot[i];
        if (i < warp) before += s;
        tot += s;
    }
    *total = tot;
    return before + incl - v;
}

template <int ELEM, int TM>
__global__ void __launch_bounds__(kThreads)
spmm_generic_kernel(const UsKParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int BITS = (ELEM == US_F16) ? 16 : (ELEM == US_I4 ? 4 : 2);   // int2: W2A4
    constexpr int E16 = 128 / BITS;
    constexpr int G = kThreads / TM;                  // token groups
    constexpr int R = kTB / G;                        // tokens per thread
    using acc_t = typename std::conditional<ELEM == US_F16, float, int>::type;

    const int TK = p.TK;
    const int Q = p.ie_ra * p.ie_ca;                  // value streams per tile (1: plain format)
    const int LM = TM / p.ie_ra, LK = TK / p.ie_ca;   // logical union-mask rows and columns
    const bool ie = Q > 1 || p.perm != nullptr;
    const int nw = TM * TK / (64 * Q);
    const int npos = TM * TK;
    const int band = blockIdx.x % p.nTM;
    const int slice = blockIdx.x / p.nTM;
    const int tb = blockIdx.y;
    const int kt0 = (int)((int64_t)slice * p.nTK / p.split);
    const int kt1 = (int)((int64_t)(slice + 1) * p.nTK / p.split);
    const int nk = kt1 - kt0;

    // ---- shared memory carve-up
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);                 // 2 barriers
    uint32_t* stage_len = reinterpret_cast<uint32_t*>(smem + 16);      // 2 run lengths (elements)
    uint32_t off = 32;
    uint32_t* offs = reinterpret_cast<uint32_t*>(smem + off);
    off = align16(off + (uint32_t)(nk + 1) * 4u);
    const uint32_t bm_bytes = (uint32_t)npos / (8u * (uint32_t)Q);
    const uint32_t val_cap = (uint32_t)npos * BITS / 8u;
    uint8_t* stage_ptr[2];
    stage_ptr[0] = smem + off; off += align16(bm_bytes + val_cap);
    stage_ptr[1] = smem + off; off += align16(bm_bytes + val_cap);
    uint32_t* wpre = reinterpret_cast<uint32_t*>(smem + off); off = align16(off + (uint32_t)nw * 4u);
    uint8_t* dense = smem + off; off = align16(off + (uint32_t)npos * (ELEM == US_F16 ? 2u : 1u));
    uint8_t* xs = smem + off;    // kTB x TK (float for F16, int8 for I4)
    __shared__ uint32_t warp_tot[kThreads / 32];
    __shared__ int flag_s;
    __shared__ uint8_t perm_s[TM];                    // the tile's row permutation (IE-BME)

    const int64_t tile0 = (int64_t)band * p.nTK + kt0;
    for (int q = threadIdx.x; q <= nk; q += kThreads) offs[q] = p.tile_off[tile0 + q];
    if (threadIdx.x == 0) {
        us::mbar_init(&bar[0], 1);
        us::mbar_init(&bar[1], 1);
        us::fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](int q) {        // thread 0 only
        const int s = q & 1;
        const uint32_t o0 = offs[q], o1 = offs[q + 1];
        const bool ok = o1 >= o0 && (o1 - o0) <= (uint32_t)npos && (o0 % E16) == 0 && (o1 % E16) == 0 &&
                        (uint64_t)o1 * BITS <= p.values_bytes * 8ull;
        const uint32_t vbytes = ok ? (o1 - o0) * BITS / 8u : 0u;
        if (!ok) us::set_status(p.status, US_ERR_CORRUPT);
        stage_len[s] = ok ? (o1 - o0) : 0u;
        us::mbar_arrive_expect_tx(&bar[s], bm_bytes + vbytes);
        us::bulk_g2s(stage_ptr[s], p.bitmap + (tile0 + q) * nw, bm_bytes, &bar[s]);
        if (vbytes) us::bulk_g2s(stage_ptr[s] + bm_bytes, p.values + (uint64_t)o0 * BITS / 8u, vbytes, &bar[s]);
    };
    if (threadIdx.x == 0) {
        if (nk > 0) issue(0);
        if (nk > 1) issue(1);
    }

    const int i_row = threadIdx.x % TM;
    const int g = threadIdx.x / TM;
    acc_t acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0;

    uint32_t phase = 0;
    for (int q = 0; q < nk; ++q) {
        const int s = q & 1;
        const bool ok = us::mbar_wait(&bar[s], (phase >> s) & 1u, p.status);
        phase ^= 1u << s;
        if (__syncthreads_or(!ok)) {
            // a copy did not land in time: give the copies in flight one more
            // bounded wait so that none is still writing when the CTA exits
            if (threadIdx.x == 0) us::mbar_wait(&bar[s ^ 1], (phase >> (s ^ 1)) & 1u, nullptr);
            return;
        }
        const uint64_t* words = reinterpret_cast<const uint64_t*>(stage_ptr[s]);
        const uint8_t* run = stage_ptr[s] + bm_bytes;
        const uint32_t len = stage_len[s];

        // 1. word prefix (nw <= 512: two words per thread)
        const int w0 = 2 * threadIdx.x, w1 = w0 + 1;
        const uint32_t c0 = (w0 < nw) ? (uint32_t)__popcll(words[w0]) : 0u;
        const uint32_t c1 = (w1 < nw) ? (uint32_t)__popcll(words[w1]) : 0u;
        uint32_t P;
        const uint32_t ex = block_excl_scan(c0 + c1, warp_tot, &P);
        if (w0 < nw) wpre[w0] = ex;
        if (w1 < nw) wpre[w1] = ex + c0;
        // activations of this K tile for this token block
        const int kbase = (kt0 + q) * TK;
        for (int idx = threadIdx.x; idx < kTB * TK; idx += kThreads) {
            const int n = idx / TK, j = idx - n * TK;
            const int ng = tb * kTB + n;
            if (ELEM == US_F16) {
                float v = 0.f;
                if (ng < p.N)
                    v = us::half_bits_to_float(reinterpret_cast<const uint16_t*>(p.X)[(int64_t)ng * p.K + kbase + j]);
                reinterpret_cast<float*>(xs)[idx] = v;
            } else {
                int8_t v = 0;
                if (ng < p.N) {
                    const uint64_t e = (uint64_t)ng * p.K + kbase + j;
                    const uint8_t by = reinterpret_cast<const uint8_t*>(p.X)[e >> 1];
                    v = (int8_t)us::sext4((e & 1) ? (by >> 4) : by);
                }
                reinterpret_cast<int8_t*>(xs)[idx] = v;
            }
        }
        if (ie && threadIdx.x < TM) {
            uint32_t r = p.perm ? p.perm[(tile0 + q) * TM + threadIdx.x] : (uint32_t)threadIdx.x;
            if (r >= (uint32_t)TM) {                  // not a row of the tile: refuse it, stay in bounds
                us::set_status(p.status, US_ERR_CORRUPT);
                r = threadIdx.x;
            }
            perm_s[threadIdx.x] = (uint8_t)r;
        }
        __syncthreads();
        const bool tile_ok = (uint64_t)P * Q <= len;
        if (!tile_ok && threadIdx.x == 0) us::set_status(p.status, US_ERR_CORRUPT);

        // 2. decode every position into the k-major dense tile
        if (ie) {
            // IE-BME with areas ("UnionSparse: An Index-Efficient Sparsity
            // Framework for Low-Bit Sparse LLM Inference on Edge", section V-A,
            // Fig. 7): position (r, k) of the reordered tile lies in area
            // q = (r / LM) * CA + k / LK at logical position (r % LM, k % LK);
            // its value is CV[o_t + q P_t + rho] if that union-mask bit is set.
            // Row r of the reordered tile is row perm[r] of the original tile.
            for (int pos = threadIdx.x; pos < npos; pos += kThreads) {
                const int r = pos / TK, k = pos - r * TK;
                const int a = r / LM, i = r - a * LM, c = k / LK, j = k - c * LK;
                const int lp = i * LK + j;
                const uint64_t word = words[lp >> 6];
                const int b = lp & 63;
                const bool set = tile_ok && ((word >> b) & 1ull);
                uint32_t e = 0;
                if (set) e = (uint32_t)(a * p.ie_ca + c) * P + wpre[lp >> 6] + (uint32_t)__popcll(word & ((1ull << b) - 1ull));
                const int row = perm_s[r];
                if (ELEM == US_F16) {
                    const uint16_t h = set ? reinterpret_cast<const uint16_t*>(run)[e] : (uint16_t)0;
                    reinterpret_cast<uint16_t*>(dense)[k * TM + row] = h;
                } else {
                    int8_t v = 0;
                    if (set) {
                        const uint8_t by = run[e >> 1];
                        v = (int8_t)us::sext4((e & 1) ? (by >> 4) : by);
                    }
                    reinterpret_cast<int8_t*>(dense)[k * TM + row] = v;
                }
            }
        } else
        for (int pos = threadIdx.x; pos < npos; pos += kThreads) {
            const int w = pos >> 6, b = pos & 63;
            const uint64_t word = words[w];
            // ROW scan p = i TK + j (IE-BME); COL scan p = j TM + i (Tiled-CBC)
            const int i = p.order == US_ORDER_COL ? pos % TM : pos / TK;
            const int j = p.order == US_ORDER_COL ? pos / TM : pos - i * TK;
            const bool set = tile_ok && ((word >> b) & 1ull);
            uint32_t rank = 0;
            if (set) rank = wpre[w] + (uint32_t)__popcll(word & ((1ull << b) - 1ull));
            if (ELEM == US_F16) {
                const uint16_t h = set ? reinterpret_cast<const uint16_t*>(run)[rank] : (uint16_t)0;
                reinterpret_cast<uint16_t*>(dense)[j * TM + i] = h;
            } else {
                int8_t v = 0;
                if (set) {
                    if (ELEM == US_I4) {
                        const uint8_t by = run[rank >> 1];
                        v = (int8_t)us::sext4((rank & 1) ? (by >> 4) : by);
                    } else {                          // int2, four per byte, earlier in the lower bits
                        const uint32_t c = (run[rank >> 2] >> (2 * (rank & 3))) & 3u;
                        v = (int8_t)((int)c - ((int)(c & 2u) << 1));
                    }
                }
                reinterpret_cast<int8_t*>(dense)[j * TM + i] = v;
            }
        }
        __syncthreads();
        if (threadIdx.x == 0 && q + 2 < nk) issue(q + 2);   // stage s is free again

        // 3. multiply
        for (int j = 0; j < TK; ++j) {
            if (ELEM == US_F16) {
                const float w = us::half_bits_to_float(reinterpret_cast<const uint16_t*>(dense)[j * TM + i_row]);
                const float* xj = reinterpret_cast<const float*>(xs) + j;
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r] = fmaf(w, xj[(g + r * G) * TK], acc[r]);
            } else {
                const int w = reinterpret_cast<const int8_t*>(dense)[j * TM + i_row];
                const int8_t* xj = reinterpret_cast<const int8_t*>(xs) + j;
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r] += w * (int)xj[(g + r * G) * TK];
            }
        }
        __syncthreads();
    }

    // ---- epilogue (split-K reduction by the last CTA of the band)
    const int m = band * TM + i_row;
    const int nTB = gridDim.y;
    if (p.split > 1) {
        acc_t* part = reinterpret_cast<acc_t*>(p.ws);
        const int64_t base = (((int64_t)slice * nTB + tb) * p.nTM + band) * (int64_t)kTB * TM;
#pragma unroll
        for (int r = 0; r < R; ++r) part[base + (int64_t)(g + r * G) * TM + i_row] = acc[r];
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned old = atomicAdd(&p.counters[band * nTB + tb], 1u);
            flag_s = (old == (unsigned)p.split - 1u);
        }
        __syncthreads();
        if (!flag_s) return;
        __threadfence();
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] = 0;
        for (int sl = 0; sl < p.split; ++sl) {
            const int64_t b2 = (((int64_t)sl * nTB + tb) * p.nTM + band) * (int64_t)kTB * TM;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                acc_t* src = part + b2 + (g + r * G) * TM + i_row;
                acc[r] += __ldcg(src);
                __stcg(src, (acc_t)0);          // leave the workspace zeroed for the next call
            }
        }
        if (threadIdx.x == 0) p.counters[band * nTB + tb] = 0u;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int n = tb * kTB + g + r * G;
        if (n >= p.N) continue;
        const int64_t o = (int64_t)n * p.M + m;
        if (ELEM == US_F16) {
            p.Y[o] = us::float_to_half_bits((float)acc[r]);
        } else {
            p.Yacc[o] = (int)acc[r];
            if (p.Y) {
                const float a = __int2float_rn((int)acc[r]);
                const float t = __fmul_rn(a, us::half_bits_to_float(p.s_w[m]));
                p.Y[o] = us::float_to_half_bits(__fmul_rn(t, us::half_bits_to_float(p.s_x[n])));
            }
        }
    }
}

size_t generic_smem(int TM, int TK, int elem, int nk) {
    const size_t npos = (size_t)TM * TK;
    const size_t bits = elem == US_F16 ? 16 : (elem == US_I4 ? 4 : 2);
    auto a16 = [](size_t x) { return (x + 15) & ~(size_t)15; };
    size_t off = 32;
    off = a16(off + (size_t)(nk + 1) * 4);
    off += 2 * a16(npos / 8 + npos * bits / 8);
    off = a16(off + (npos / 64) * 4);
    off = a16(off + npos * (elem == US_F16 ? 2 : 1));
    off += (size_t)kTB * TK * (elem == US_F16 ? 4 : 1);
    return off;
}

template <int ELEM, int TM>
us_status launch_t(const UsKParams& p, cudaStream_t st) {
    const int nk = (p.nTK + p.split - 1) / p.split;
    const size_t smem = generic_smem(TM, p.TK, ELEM, nk);
    if (smem > 227 * 1024) return US_ERR_UNSUPPORTED;
    auto kern = spmm_generic_kernel<ELEM, TM>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return US_ERR_CUDA;
    dim3 grid((unsigned)(p.nTM * p.split), (unsigned)((p.N + kTB - 1) / kTB));
    kern<<<grid, kThreads, smem, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? US_OK : US_ERR_CUDA;
}

}  // namespace

namespace us {

int spmm_generic_tok_block(int) { return kTB; }

size_t spmm_generic_ws(int M, int TM, int N, int split, int tok_block) {
    const int nTM = M / TM;
    const int nTB = (N + tok_block - 1) / tok_block;
    const size_t counters = ((size_t)nTM * nTB * 4 + 255) & ~(size_t)255;
    if (split <= 1) return counters;
    return counters + (size_t)split * nTB * nTM * tok_block * TM * 4;
}

us_status launch_spmm_generic(const UsKParams& p, int elem, cudaStream_t st) {
    if (elem == US_F16) {
        switch (p.TM) {
            case 16: return launch_t<US_F16, 16>(p, st);
            case 64: return launch_t<US_F16, 64>(p, st);
            case 128: return launch_t<US_F16, 128>(p, st);
            case 256: return launch_t<US_F16, 256>(p, st);
        }
    } else if (elem == US_I2) {
        switch (p.TM) {
            case 64: return launch_t<US_I2, 64>(p, st);
            case 128: return launch_t<US_I2, 128>(p, st);
            case 256: return launch_t<US_I2, 256>(p, st);
        }
    } else {
        switch (p.TM) {
            case 16: return launch_t<US_I4, 16>(p, st);
            case 64: return launch_t<US_I4, 64>(p, st);
            case 128: return launch_t<US_I4, 128>(p, st);
            case 256: return launch_t<US_I4, 256>(p, st);
        }
    }
    return US_ERR_UNSUPPORTED;
}

}  // namespace us
