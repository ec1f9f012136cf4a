// us_common.cuh -- device helpers shared by the libus kernels (sm_103a).
//
// Inline PTX for the Blackwell data movers used by every kernel: mbarrier
// transaction barriers and the bulk (TMA 1-D) global->shared copy, plus the
// bounded waits and the device status word that replace traps and endless
// spins.  Nothing here belongs to the format's arithmetic.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "../../include/us.h"

#define US_DEV __device__ __forceinline__

namespace us {

// ----------------------------------------------------------------- status --
// The first device-side error wins; later ones are dropped.
US_DEV void set_status(unsigned* status, unsigned code) {
    if (status) atomicCAS(status, 0u, code);
}

US_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// A wait gives up after this long; the kernel then records US_ERR_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s

// --------------------------------------------------------------- mbarrier --
US_DEV uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

US_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

US_DEV void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

US_DEV void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

US_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

US_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// `count` arrivals at once
US_DEV void mbar_arrive_n(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

US_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of `bar`.  Returns false (and records
// US_ERR_TIMEOUT) if the phase did not complete within kWaitLimitNs.
// As mbar_try_wait, but the thread may sleep up to `ns` for the phase first.
US_DEV bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// As mbar_wait, with the limit given in nanoseconds.
US_DEV bool mbar_wait_for(uint64_t* bar, uint32_t parity, unsigned* status, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, parity, 100000u)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            set_status(status, US_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

US_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* status) {
    return mbar_wait_for(bar, parity, status, kWaitLimitNs);
}


// Bulk copy global -> shared (TMA, 1-D, no tensor map), completing `bytes`
// transactions on `bar`.  dst, src 16-byte aligned; bytes a multiple of 16.
US_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// L2 prefetch of a global range (bytes a multiple of 16).
US_DEV void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ------------------------------------------- programmatic dependent launch --
// A kernel launched with programmatic stream serialisation may start while
// its predecessor drains; it must not read anything a predecessor could have
// written before pdl_wait(), which returns once every prerequisite grid has
// completed and its memory is visible.  pdl_launch_dependents() lets the next
// such kernel start its own prologue early.  Both are no-ops for ordinary
// launches.
US_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
US_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// One three-input logic op: bit i of the result is bit (a_i b_i c_i) of LUT,
// the truth table over a = 0xF0, b = 0xCC, c = 0xAA.  Written out because
// the compiler does not always merge a mask-and-combine into one.
template <uint32_t LUT>
US_DEV uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(d) : "r"(a), "r"(b), "r"(c), "n"(LUT));
    return d;
}
constexpr uint32_t kLopAndXor = (0xF0u & 0xCCu) ^ 0xAAu;                  // (a & b) ^ c
constexpr uint32_t kLopMux = (0xF0u & 0xCCu) | (0xAAu & ~0xCCu & 0xFFu);   // (a & b) | (c & ~b)

// Named barrier over the first `threads` threads (a multiple of 32), id 1..15.
US_DEV void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- clusters --
US_DEV uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster must call this (hardware barrier).
US_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of `p` (this CTA's shared memory) in the shared memory of cluster CTA `rank`.
US_DEV uint32_t cluster_map(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}
// 64-bit global word, relaxed at GPU scope: single-copy atomic, never served
// from a stale L1 line.  Used for {value, tag} messages between CTAs.
US_DEV uint64_t ld_relaxed_gpu_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
US_DEV void st_relaxed_gpu_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

US_DEV int ld_cluster_s32(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
US_DEV float4 ld_cluster_v4f32(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}
US_DEV float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// ------------------------------------------------------------------- misc --
US_DEV uint32_t lane_id() { return threadIdx.x & 31u; }

US_DEV int warp_incl_scan(int v) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, v, d);
        if ((int)lane_id() >= d) v += o;
    }
    return v;
}

US_DEV float half_bits_to_float(uint16_t h) { return __half2float(__ushort_as_half(h)); }
US_DEV uint16_t float_to_half_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }

// int4 code in the low nibble of v -> int (two's complement)
US_DEV int sext4(uint32_t v) { return (int)(v << 28) >> 28; }

// PTX shl clamps shift counts >= 32 to a zero result (C++ leaves them undefined)
US_DEV uint32_t shl_clamp(uint32_t x, uint32_t n) {
    uint32_t r;
    asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(n));
    return r;
}

// v = shared-memory word at `addr` if `pred`, else v unchanged (a predicated
// load: lanes with pred == 0 touch no bank).  volatile keeps it in program
// order with the mbarrier operations around it.
US_DEV void lds_u32_if(uint32_t& v, uint32_t pred, uint32_t addr) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t@p ld.shared.u32 %0, [%2];\n\t}"
        : "+r"(v)
        : "r"(pred), "r"(addr));
}

// Bytes (w + 8) of ranks 0,2,4,6 (even) and 1,3,5,7 (odd) -> eight fp16 values
// at the positions the PRMT selector pair names: 0x6400 | (w + 8) is the fp16
// number 1024 + w + 8, minus 1032 leaves w exactly.
US_DEV uint4 u8x8_to_f16x8(uint32_t even, uint32_t odd, uint32_t sel) {
    const uint32_t d0 = __byte_perm(even, odd, sel);
    const uint32_t d1 = __byte_perm(even, odd, sel >> 16);
    const uint32_t k64 = 0x64646464u;
    const uint32_t b[4] = {__byte_perm(d0, k64, 0x5140), __byte_perm(d0, k64, 0x7362),
                           __byte_perm(d1, k64, 0x5140), __byte_perm(d1, k64, 0x7362)};
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&b[i]), bias);
        o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// d += A . B for one m16n8k16 tile: fp16 A (row-major fragment a0..a3), fp16 B
// (column-major fragment b0, b1), fp32 accumulators.
US_DEV void mma_m16n8k16_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte-step decode of packed int4 runs (used by the W4A4 kernels).  For one
// bitmap byte v (8 positions) the run's next popc(v) nibbles are split into
// even and odd ranks, one byte each; make_sel(v) is the PRMT selector pair
// that moves rank r to its position p: byte r/2 of the even register or
// 4 + r/2 of the odd one.  Clear positions take byte 7 (rank 7), which the
// masked window leaves empty unless all eight positions are set.  Low 16 bits
// cover positions 0-3, high 16 bits positions 4-7.
__host__ __device__ constexpr uint32_t make_sel(uint32_t v) {
    uint32_t sel = 0, r = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const uint32_t set = (v >> p) & 1u;
        const uint32_t idx = set ? ((r & 1u) ? 4u + (r >> 1) : (r >> 1)) : 7u;
        sel |= idx << (4 * (p & 3) + 16 * (p >> 2));
        r += set;
    }
    return sel;
}

}  // namespace us

// ------------------------------------------------------- kernel parameters --
// One plain struct passed by value to every SpMM / spMspV kernel.
struct UsKParams {
    int M, K, TM, TK, nTM, nTK;
    int N;              // tokens
    int split;          // K slices
    int tok_block;      // tokens per CTA (grid.y = ceil(N / tok_block))
    const uint64_t* bitmap;
    const uint32_t* tile_off;
    const uint8_t* values;
    uint64_t values_bytes;
    const void* X;      // I4: packed nibbles N x K; F16: fp16 N x K
    const uint16_t* s_w;
    const uint16_t* s_x;
    int32_t* Yacc;
    uint16_t* Y;
    float tau;
    uint32_t flags;     // US_BITMAP_* flags of the weight descriptor
    int order;          // US_ORDER_ROW or US_ORDER_COL scan inside a tile
    // IE-BME with areas (generic kernel only): RA row x CA column partitions of
    // each tile, one union mask, Q = RA*CA value streams; perm: per tile, the
    // original row of each row of the reordered tile (nullptr = identity)
    int elem;           // US_F16, US_I4 or US_I2 values
    int ie_ra, ie_ca;
    const uint8_t* perm;
    void* ws;           // split-K partials (after the counters)
    unsigned* counters; // split-K arrival counters, one per (band, token block)
    unsigned* status;
    // balanced (stream-K) W4A4 kernel only: CTAs, most tiles of one CTA, value
    // ring bytes, staged activation columns (tiles), most bands one CTA touches,
    // dense decoded-tile slots, tiles decoded before the dependency wait
    int sk_grid, sk_per, sk_ring, sk_xcols, sk_nb, sk_slots, sk_pre;
};
