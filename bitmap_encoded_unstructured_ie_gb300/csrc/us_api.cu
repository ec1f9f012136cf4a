// us_api.cu -- the C ABI of libus: argument checks, sizes, dispatch.
//
// Every entry point validates on the host before enqueuing anything and
// returns a us_status; nothing throws across the ABI.  The device status word
// g_us_status collects device-side errors (timeouts, corrupt offsets,
// out-of-range codes); us_get_last_device_status reads and clears it.
#include <mutex>

#include "us_common.cuh"
#include "us_internal.h"

__device__ unsigned g_us_status = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return (d >= 0 && d < kMaxDevices) ? d : -1;
}

// Device address of g_us_status on the current device (looked up once).
unsigned* status_ptr() {
    const int d = current_device();
    if (d < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[d]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_us_status) != cudaSuccess) return nullptr;
        g_status_ptr[d] = static_cast<unsigned*>(p);
    }
    return g_status_ptr[d];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool tile_ok(int TM, int TK) {
    return (TM == 64 || TM == 128 || TM == 256) && (TK == 16 || TK == 32 || TK == 64 || TK == 128);
}

us_status check_shape(int M, int K, int TM, int TK, int elem) {
    if (M <= 0 || K <= 0 || !tile_ok(TM, TK)) return US_ERR_INVALID_ARG;
    if (M % TM || K % TK) return US_ERR_INVALID_ARG;
    if (elem != US_F16 && elem != US_I4 && elem != US_I2) return US_ERR_INVALID_ARG;
    if ((uint64_t)M * (uint64_t)K >= (1ull << 32)) return US_ERR_TOO_LARGE;
    return US_OK;
}

us_status check_bitmap(const us_bitmap* W, int elem, int order) {
    if (!W) return US_ERR_INVALID_ARG;
    us_status s = check_shape(W->M, W->K, W->TM, W->TK, W->elem);
    if (s != US_OK) return s;
    if (W->order != US_ORDER_ROW && W->order != US_ORDER_COL) return US_ERR_INVALID_ARG;
    if (W->elem != elem) return US_ERR_INVALID_ARG;
    if (W->order != order) return US_ERR_UNSUPPORTED;
    if (!W->bitmap || !W->tile_off || (!W->values && W->values_bytes)) return US_ERR_INVALID_ARG;
    if (!aligned16(W->bitmap) || !aligned16(W->tile_off) || !aligned16(W->values)) return US_ERR_INVALID_ARG;
    if ((W->flags & ~US_BITMAP_STATIC) || W->reserved) return US_ERR_INVALID_ARG;
    return US_OK;
}

// split-K rule: the smallest candidate whose grid covers every SM, keeping at
// least 4 K tiles per slice.
int auto_split(int nTM, int nTK, int token_blocks, int target = 0, int max_split = 16) {
    const int sms = target > 0 ? target : us::num_sms();
    const int cands[] = {1, 2, 4, 8, 16};
    int best = 1;
    for (int c : cands) {
        if (nTK / c < 4 || c > max_split) break;
        best = c;
        if ((int64_t)nTM * c * token_blocks >= sms) break;
    }
    return best;
}

void fill_common(UsKParams& p, const us_bitmap* W, int N) {
    p.M = W->M; p.K = W->K; p.TM = W->TM; p.TK = W->TK;
    p.nTM = W->M / W->TM; p.nTK = W->K / W->TK;
    p.N = N;
    p.bitmap = W->bitmap; p.tile_off = W->tile_off;
    p.values = static_cast<const uint8_t*>(W->values);
    p.values_bytes = W->values_bytes;
    p.X = nullptr; p.s_w = nullptr; p.s_x = nullptr; p.Yacc = nullptr; p.Y = nullptr;
    p.tau = 0.f; p.ws = nullptr; p.counters = nullptr;
    p.sk_grid = p.sk_per = p.sk_ring = p.sk_xcols = p.sk_nb = p.sk_slots = p.sk_pre = 0;
    p.flags = W->flags;
    p.order = W->order;
    p.elem = W->elem;
    p.ie_ra = p.ie_ca = 1;
    p.perm = nullptr;
    p.status = status_ptr();
}

// Launch plan for an SpMM call: kernel family, split, token block, workspace.
struct Plan {
    bool sk;        // W4A4 CUDA-core kernel over a balanced partition of the tiles
    bool fast;      // W4A4 register-decode kernel
    bool tc;        // fp16 tensor-core kernel
    bool dec;       // fp16 decode kernel (1-63 tokens, mma.sync)
    int split;
    int tok_block;
    size_t ws;
};

Plan plan_spmm(us_op op, const us_bitmap* W, int N, int split_k) {
    Plan pl{};
    // W4A4, automatic split: the balanced kernels (no K slices; tiles spread
    // evenly over the SMs)
    if (op == US_OP_SPMM_W4A4 && split_k == 0) {
        if (us::w4a4_sk_supported(W->TM, W->TK, W->M, W->K, N)) {
            pl.sk = true;
            pl.tok_block = N;
            pl.ws = us::w4a4_sk_ws(W->M, W->K, N);
            return pl;
        }
    }
    if (op == US_OP_SPMM_F16 && us::tc_f16_supported(W->TM, W->TK, W->M, N)) {
        pl.tc = true;
        pl.tok_block = us::tc_tok_block(N);
        pl.split = split_k > 0 ? split_k : us::tc_split(W->M, N, W->K / W->TK);
        if (pl.split > W->K / W->TK) pl.split = W->K / W->TK;
        if (pl.split > us::tc_max_split()) pl.split = us::tc_max_split();
        pl.ws = us::tc_ws(W->M, N, pl.split);
        return pl;
    }
    const int nTM = W->M / W->TM, nTK = W->K / W->TK;
    if (op == US_OP_SPMM_F16 && us::f16_dec_supported(W->TM, W->TK, W->order, N) &&
        (split_k == 0 || us::f16_dec_fits(nTK, split_k, N))) {
        pl.dec = true;
        pl.tok_block = us::f16_dec_tok_block(N);
        pl.split = split_k > 0 ? split_k : us::f16_dec_split(nTM, nTK, N);
        pl.ws = us::spmm_generic_ws(W->M, W->TM, N, pl.split, pl.tok_block);
        return pl;
    }
    pl.fast = (op == US_OP_SPMM_W4A4) && W->elem == US_I4 && us::w4a4_fast_supported(W->TM, W->TK, N) &&
              split_k <= us::w4a4_fast_max_split();
    pl.tok_block = pl.fast ? us::w4a4_fast_tok_block(N) : us::spmm_generic_tok_block(N);
    const int ntb = (N + pl.tok_block - 1) / pl.tok_block;
    pl.split = split_k > 0 ? split_k
                           : auto_split(nTM, nTK, ntb, pl.fast ? us::w4a4_fast_target_ctas() : 0,
                                        pl.fast ? us::w4a4_fast_max_split() : 16);
    if (pl.split > nTK) pl.split = nTK;
    pl.ws = pl.fast ? us::w4a4_fast_ws(W->M, W->TM, N, pl.split)
                    : us::spmm_generic_ws(W->M, W->TM, N, pl.split, pl.tok_block);
    return pl;
}

// streamed: us_spmspv_f16 may take the streamed kernel (64 x 64 tiles); the
// batched ColInfo kernel plans with streamed = false
Plan plan_spmspv(const us_bitmap* W, bool streamed = true) {
    Plan pl{};
    pl.tok_block = 1;
    const int ss = streamed ? us::spmspv_stream_split(W->TM, W->TK, W->M / W->TM, W->K / W->TK) : 0;
    if (ss > 0) {
        pl.dec = true;                    // the streamed kernel
        pl.split = ss;
        return pl;
    }
    pl.split = auto_split(W->M / W->TM, W->K / W->TK, 1, 2 * us::num_sms(), us::spmspv_max_split());
    pl.ws = us::spmspv_ws(W->M, W->TM, pl.split);
    return pl;
}

size_t counters_bytes(int nTM, int ntb) { return ((size_t)nTM * ntb * 4 + 255) & ~(size_t)255; }

}  // namespace

namespace us {

int num_sms() {
    const int d = current_device();
    if (d < 0) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_num_sms[d]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || v <= 0) v = 148;
        g_num_sms[d] = v;
    }
    return g_num_sms[d];
}

}  // namespace us

namespace {

// One thread waits on an mbarrier that nothing arrives on (no copy or other
// asynchronous operation is in flight), through the same bounded wait every
// kernel uses, with the caller's limit.
__global__ void wait_selftest_kernel(unsigned* status, uint64_t limit_ns, uint64_t* elapsed_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    us::mbar_init(&bar, 1);
    us::fence_mbar_init();
    const uint64_t t0 = us::globaltimer_ns();
    const bool done = us::mbar_wait_for(&bar, 0u, status, limit_ns);
    if (elapsed_ns) *elapsed_ns = done ? 0ull : us::globaltimer_ns() - t0;
}

}  // namespace

extern "C" {

int us_version(void) { return 100; }

const char* us_status_string(us_status s) {
    switch (s) {
        case US_OK: return "ok";
        case US_ERR_INVALID_ARG: return "invalid argument";
        case US_ERR_UNSUPPORTED: return "unsupported combination";
        case US_ERR_TOO_LARGE: return "too large";
        case US_ERR_WORKSPACE: return "workspace or capacity too small";
        case US_ERR_CUDA: return "CUDA error";
        case US_ERR_TIMEOUT: return "device wait timed out";
        case US_ERR_CORRUPT: return "corrupt format";
    }
    return "unknown status";
}

us_status us_encode_sizes(int M, int K, int TM, int TK, us_elem elem, size_t* bitmap_bytes,
                          size_t* tile_off_bytes, size_t* values_cap_bytes, size_t* ws_bytes) {
    us_status s = check_shape(M, K, TM, TK, elem);
    if (s != US_OK) return s;
    const uint64_t nT = (uint64_t)(M / TM) * (K / TK);
    if (bitmap_bytes) *bitmap_bytes = (size_t)M * K / 8;
    if (tile_off_bytes) *tile_off_bytes = (size_t)(nT + 1) * 4;
    if (values_cap_bytes) *values_cap_bytes = (size_t)M * K * (elem == US_F16 ? 16 : (elem == US_I4 ? 4 : 2)) / 8;
    if (ws_bytes) *ws_bytes = ((size_t)nT * 4 + 255) & ~(size_t)255;
    return US_OK;
}

us_status us_encode(const void* W, int64_t ldw, int M, int K, int TM, int TK, us_elem elem, us_order order,
                    uint64_t* bitmap, uint32_t* tile_off, void* values, size_t values_cap, void* ws,
                    size_t ws_bytes, void* stream) {
    us_status s = check_shape(M, K, TM, TK, elem);
    if (s != US_OK) return s;
    if (order != US_ORDER_ROW && order != US_ORDER_COL) return US_ERR_INVALID_ARG;
    if (!W || !bitmap || !tile_off || !values || !ws || ldw < K) return US_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & (elem == US_F16 ? 1u : 0u)) != 0) return US_ERR_INVALID_ARG;
    if (!aligned16(bitmap) || !aligned16(tile_off) || !aligned16(values) || !aligned16(ws))
        return US_ERR_INVALID_ARG;
    size_t need = 0;
    us_encode_sizes(M, K, TM, TK, elem, nullptr, nullptr, nullptr, &need);
    if (ws_bytes < need) return US_ERR_WORKSPACE;
    return us::launch_encode(W, ldw, M, K, TM, TK, elem, order, bitmap, tile_off, values, values_cap,
                             static_cast<uint32_t*>(ws), status_ptr(), static_cast<cudaStream_t>(stream));
}

us_status us_workspace_bytes(us_op op, const us_bitmap* W, int N, int split_k, size_t* bytes) {
    if (!W || !bytes) return US_ERR_INVALID_ARG;
    us_status s = check_shape(W->M, W->K, W->TM, W->TK, op == US_OP_ENCODE ? US_F16 : W->elem);
    if (s != US_OK) return s;
    if (split_k < 0) return US_ERR_INVALID_ARG;
    switch (op) {
        case US_OP_ENCODE:
            return us_encode_sizes(W->M, W->K, W->TM, W->TK, US_F16, nullptr, nullptr, nullptr, bytes);
        case US_OP_SPMM_W4A4:
        case US_OP_SPMM_F16:
            if (N < 1 || N > 2048) return US_ERR_INVALID_ARG;
            *bytes = plan_spmm(op, W, N, split_k).ws;
            return US_OK;
        case US_OP_SPMSPV_F16: {
            Plan pl = plan_spmspv(W);
            if (split_k > 0) pl.ws = us::spmspv_ws(W->M, W->TM, split_k);
            *bytes = pl.ws;
            return US_OK;
        }
    }
    return US_ERR_INVALID_ARG;
}

us_status us_pick_split_k(us_op op, const us_bitmap* W, int N, int* split_k) {
    if (!W || !split_k) return US_ERR_INVALID_ARG;
    us_status s = check_shape(W->M, W->K, W->TM, W->TK, W->elem);
    if (s != US_OK) return s;
    if (op == US_OP_SPMSPV_F16) { *split_k = plan_spmspv(W).split; return US_OK; }
    if (op != US_OP_SPMM_W4A4 && op != US_OP_SPMM_F16) return US_ERR_INVALID_ARG;
    if (N < 1 || N > 2048) return US_ERR_INVALID_ARG;
    *split_k = plan_spmm(op, W, N, 0).split;
    return US_OK;
}

us_status us_spmm_w4a4(const us_bitmap* W, const uint8_t* Xq, const uint16_t* s_w, const uint16_t* s_x, int N,
                       int32_t* Yacc, uint16_t* Y, void* ws, size_t ws_bytes, int split_k, void* stream) {
    // W4A4, or W2A4 with int2 weights
    us_status s = check_bitmap(W, W && W->elem == US_I2 ? US_I2 : US_I4, US_ORDER_ROW);
    if (s != US_OK) return s;
    if (N < 1 || N > 2048 || W->K % 32) return US_ERR_INVALID_ARG;
    if (!Xq || !Yacc || !aligned16(Xq) || !aligned16(Yacc)) return US_ERR_INVALID_ARG;
    if (Y && (!s_w || !s_x || !aligned16(Y))) return US_ERR_INVALID_ARG;
    if (split_k < 0 || split_k > W->K / W->TK) return US_ERR_INVALID_ARG;
    const Plan pl = plan_spmm(US_OP_SPMM_W4A4, W, N, split_k);
    if (pl.ws && (!ws || ws_bytes < pl.ws || !aligned16(ws))) return US_ERR_WORKSPACE;
    UsKParams p;
    fill_common(p, W, N);
    p.X = Xq; p.s_w = s_w; p.s_x = s_x; p.Yacc = Yacc; p.Y = Y;
    p.split = pl.split; p.tok_block = pl.tok_block;
    const int ntb = (N + pl.tok_block - 1) / pl.tok_block;
    p.counters = static_cast<unsigned*>(ws);
    p.ws = static_cast<uint8_t*>(ws) + counters_bytes(p.nTM, ntb);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (pl.sk) {
        p.ws = ws;
        return us::launch_w4a4_sk(p, st);
    }
    return pl.fast ? us::launch_w4a4_fast(p, st) : us::launch_spmm_generic(p, W->elem, st);
}

us_status us_spmm_f16(const us_bitmap* W, const uint16_t* X, int N, uint16_t* Y, void* ws, size_t ws_bytes,
                      int split_k, void* stream) {
    // either scan order: ROW (IE-BME) or COL (Tiled-CBC, the spMspV format)
    us_status s = check_bitmap(W, US_F16, W && W->order == US_ORDER_COL ? US_ORDER_COL : US_ORDER_ROW);
    if (s != US_OK) return s;
    if (N < 1 || N > 2048) return US_ERR_INVALID_ARG;
    if (!X || !Y || !aligned16(X) || !aligned16(Y)) return US_ERR_INVALID_ARG;
    if (split_k < 0 || split_k > W->K / W->TK) return US_ERR_INVALID_ARG;
    if (!ws) return US_ERR_WORKSPACE;
    const Plan pl = plan_spmm(US_OP_SPMM_F16, W, N, split_k);
    if (ws_bytes < pl.ws || !aligned16(ws)) return US_ERR_WORKSPACE;
    UsKParams p;
    fill_common(p, W, N);
    p.X = X; p.Y = Y;
    p.split = pl.split; p.tok_block = pl.tok_block;
    const int ntb = (N + pl.tok_block - 1) / pl.tok_block;
    p.counters = static_cast<unsigned*>(ws);
    if (pl.tc) return us::launch_tc_f16(p, static_cast<cudaStream_t>(stream));
    p.ws = static_cast<uint8_t*>(ws) + counters_bytes(p.nTM, ntb);
    if (pl.dec) return us::launch_f16_dec(p, static_cast<cudaStream_t>(stream));
    return us::launch_spmm_generic(p, US_F16, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------- no-allocation fp16 SpMM --
// Some callers cannot allocate device memory at the point where they multiply:
// code running while a CUDA graph is being captured (a cudaMalloc there breaks
// the capture), allocators that hand out a fixed arena, or embedders that own
// every device allocation themselves.  us_spmm_f16_noalloc serves them with
// split-K scratch that lives in this library: a file-scope device array sized
// US_NOALLOC_SCRATCH_BYTES, created when the library is loaded onto a device
// and kept until the process exits.
static __device__ __align__(256) uint8_t g_us_noalloc_scratch[US_NOALLOC_SCRATCH_BYTES];

namespace {
uint8_t* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (host code may not use the array's name as a device address).
uint8_t* noalloc_scratch_ptr() {
    const int d = current_device();
    if (d < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[d]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_us_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
        g_noalloc_ptr[d] = static_cast<uint8_t*>(ptr);
    }
    return g_noalloc_ptr[d];
}
}  // namespace

us_status us_spmm_f16_noalloc(const us_bitmap* W, const uint16_t* X, int N, uint16_t* Y, int split_k, void* stream) {
    us_status s = check_bitmap(W, US_F16, W && W->order == US_ORDER_COL ? US_ORDER_COL : US_ORDER_ROW);
    if (s != US_OK) return s;
    if (N < 1 || N > 2048) return US_ERR_INVALID_ARG;
    if (!X || !Y || !aligned16(X) || !aligned16(Y)) return US_ERR_INVALID_ARG;
    if (split_k < 0 || split_k > W->K / W->TK) return US_ERR_INVALID_ARG;
    Plan pl = plan_spmm(US_OP_SPMM_F16, W, N, split_k);
    if (pl.ws > US_NOALLOC_SCRATCH_BYTES && split_k == 0) pl = plan_spmm(US_OP_SPMM_F16, W, N, 1);
    if (pl.ws > US_NOALLOC_SCRATCH_BYTES) return US_ERR_TOO_LARGE;
    uint8_t* scratch = noalloc_scratch_ptr();
    if (!scratch) return US_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    UsKParams p;
    fill_common(p, W, N);
    p.X = X; p.Y = Y;
    p.split = pl.split; p.tok_block = pl.tok_block;
    const int ntb = (N + pl.tok_block - 1) / pl.tok_block;
    // the tensor-core path reduces its K slices inside a cluster: no scratch
    if (pl.tc) return us::launch_tc_f16(p, st);
    const size_t cbytes = counters_bytes(p.nTM, ntb);
    // the split-K arrival counters must start at zero; the partials are fully
    // written before they are read, so only the counters are cleared
    if (cudaMemsetAsync(scratch, 0, cbytes, st) != cudaSuccess) return US_ERR_CUDA;
    p.counters = reinterpret_cast<unsigned*>(scratch);
    p.ws = scratch + cbytes;
    return pl.dec ? us::launch_f16_dec(p, st) : us::launch_spmm_generic(p, US_F16, st);
}

us_status us_spmspv_f16(const us_bitmap* W, const uint16_t* x, float tau, uint16_t* y, void* ws, size_t ws_bytes,
                        void* stream) {
    us_status s = check_bitmap(W, US_F16, US_ORDER_COL);
    if (s != US_OK) return s;
    if (!x || !y || !aligned16(x) || !aligned16(y) || !(tau >= 0.f)) return US_ERR_INVALID_ARG;
    const Plan pl = plan_spmspv(W);
    if (pl.ws && (!ws || ws_bytes < pl.ws || !aligned16(ws))) return US_ERR_WORKSPACE;
    UsKParams p;
    fill_common(p, W, 1);
    p.X = x; p.Y = y; p.tau = tau;
    p.split = pl.split; p.tok_block = 1;
    p.counters = static_cast<unsigned*>(ws);
    p.ws = static_cast<uint8_t*>(ws) + counters_bytes(p.nTM, 1);
    if (pl.dec) return us::launch_spmspv_stream(p, static_cast<cudaStream_t>(stream));
    return us::launch_spmspv(p, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------- IE-BME with areas --
namespace {

us_status check_ie_shape(int M, int K, int TM, int TK, int RA, int CA, int elem) {
    if (M <= 0 || K <= 0) return US_ERR_INVALID_ARG;
    if (!(TM == 16 || TM == 64 || TM == 128 || TM == 256) || !(TK == 16 || TK == 32 || TK == 64 || TK == 128))
        return US_ERR_INVALID_ARG;
    if (!(RA == 1 || RA == 2 || RA == 4) || !(CA == 1 || CA == 2 || CA == 4) || RA * CA > 4) return US_ERR_INVALID_ARG;
    if (((TM / RA) * (TK / CA)) % 128) return US_ERR_INVALID_ARG;
    if (M % TM || K % TK) return US_ERR_INVALID_ARG;
    if (elem != US_F16 && elem != US_I4) return US_ERR_INVALID_ARG;
    if ((uint64_t)M * (uint64_t)K >= (1ull << 32)) return US_ERR_TOO_LARGE;
    return US_OK;
}

us_status check_bitmap_ie(const us_bitmap_ie* B, int elem) {
    if (!B) return US_ERR_INVALID_ARG;
    const us_bitmap* W = &B->W;
    us_status s = check_ie_shape(W->M, W->K, W->TM, W->TK, B->RA, B->CA, W->elem);
    if (s != US_OK) return s;
    if (W->elem != elem || W->order != US_ORDER_ROW) return US_ERR_INVALID_ARG;
    if (!W->bitmap || !W->tile_off || (!W->values && W->values_bytes)) return US_ERR_INVALID_ARG;
    if (!aligned16(W->bitmap) || !aligned16(W->tile_off) || !aligned16(W->values) || !aligned16(B->perm))
        return US_ERR_INVALID_ARG;
    if ((W->flags & ~US_BITMAP_STATIC) || W->reserved) return US_ERR_INVALID_ARG;
    return US_OK;
}

Plan plan_ie(const us_bitmap_ie* B, int N, int split_k) {
    Plan pl{};
    const us_bitmap* W = &B->W;
    // automatic split on 16 x 64 local tiles: the balanced kernel (no K slices)
    if (split_k == 0 && W->elem == US_I4 &&
        us::w4a4_sk_ie_supported(W->M, W->K, W->TM, W->TK, B->RA, B->CA, N)) {
        pl.sk = true;
        pl.tok_block = N;
        pl.ws = us::w4a4_sk_ie_ws(W->M, W->K, N);
        return pl;
    }
    const int nTM = W->M / W->TM, nTK = W->K / W->TK;
    pl.tok_block = us::spmm_generic_tok_block(N);
    const int ntb = (N + pl.tok_block - 1) / pl.tok_block;
    // small local tiles make thin bands: slice K deeper so that each CTA walks
    // fewer tiles (its per-tile work is short and barrier bound)
    pl.split = split_k > 0 ? split_k : auto_split(nTM, nTK, ntb, 8 * us::num_sms());
    if (pl.split > nTK) pl.split = nTK;
    pl.ws = us::spmm_generic_ws(W->M, W->TM, N, pl.split, pl.tok_block);
    return pl;
}

}  // namespace

us_status us_encode_ie_sizes(int M, int K, int TM, int TK, int RA, int CA, us_elem elem, size_t* bitmap_bytes,
                             size_t* tile_off_bytes, size_t* values_cap_bytes, size_t* ws_bytes) {
    us_status s = check_ie_shape(M, K, TM, TK, RA, CA, elem);
    if (s != US_OK) return s;
    const uint64_t nT = (uint64_t)(M / TM) * (K / TK);
    if (bitmap_bytes) *bitmap_bytes = (size_t)M * K / (8 * RA * CA);
    if (tile_off_bytes) *tile_off_bytes = (size_t)(nT + 1) * 4;
    // Q * P_t <= TM * TK per tile, and TM * TK is a multiple of the padding quantum
    if (values_cap_bytes) *values_cap_bytes = (size_t)M * K * (elem == US_F16 ? 2 : 1) / (elem == US_F16 ? 1 : 2);
    if (ws_bytes) *ws_bytes = ((size_t)nT * 4 + 255) & ~(size_t)255;
    return US_OK;
}

us_status us_encode_ie(const void* W, int64_t ldw, int M, int K, int TM, int TK, int RA, int CA, us_elem elem,
                       const uint8_t* perm, uint64_t* bitmap, uint32_t* tile_off, void* values, size_t values_cap,
                       void* ws, size_t ws_bytes, void* stream) {
    us_status s = check_ie_shape(M, K, TM, TK, RA, CA, elem);
    if (s != US_OK) return s;
    if (!W || !bitmap || !tile_off || !values || !ws || ldw < K) return US_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & (elem == US_F16 ? 1u : 0u)) != 0) return US_ERR_INVALID_ARG;
    if (!aligned16(bitmap) || !aligned16(tile_off) || !aligned16(values) || !aligned16(ws)) return US_ERR_INVALID_ARG;
    size_t need = 0;
    us_encode_ie_sizes(M, K, TM, TK, RA, CA, elem, nullptr, nullptr, nullptr, &need);
    if (ws_bytes < need) return US_ERR_WORKSPACE;
    return us::launch_encode_ie(W, ldw, M, K, TM, TK, RA, CA, elem, perm, bitmap, tile_off, values, values_cap,
                                static_cast<uint32_t*>(ws), status_ptr(), static_cast<cudaStream_t>(stream));
}

us_status us_workspace_bytes_ie(const us_bitmap_ie* B, int N, int split_k, size_t* bytes) {
    if (!B || !bytes) return US_ERR_INVALID_ARG;
    us_status s = check_ie_shape(B->W.M, B->W.K, B->W.TM, B->W.TK, B->RA, B->CA, B->W.elem);
    if (s != US_OK) return s;
    if (N < 1 || N > 2048 || split_k < 0) return US_ERR_INVALID_ARG;
    *bytes = plan_ie(B, N, split_k).ws;
    return US_OK;
}

us_status us_pick_split_k_ie(const us_bitmap_ie* B, int N, int* split_k) {
    if (!split_k) return US_ERR_INVALID_ARG;
    us_status s = check_bitmap_ie(B, US_I4);
    if (s != US_OK) return s;
    if (N < 1 || N > 2048) return US_ERR_INVALID_ARG;
    *split_k = plan_ie(B, N, 0).split;
    return US_OK;
}

us_status us_spmm_w4a4_ie(const us_bitmap_ie* B, const uint8_t* Xq, const uint16_t* s_w, const uint16_t* s_x, int N,
                          int32_t* Yacc, uint16_t* Y, void* ws, size_t ws_bytes, int split_k, void* stream) {
    us_status s = check_bitmap_ie(B, US_I4);
    if (s != US_OK) return s;
    const us_bitmap* W = &B->W;
    if (N < 1 || N > 2048 || W->K % 32) return US_ERR_INVALID_ARG;
    if (!Xq || !Yacc || !aligned16(Xq) || !aligned16(Yacc)) return US_ERR_INVALID_ARG;
    if (Y && (!s_w || !s_x || !aligned16(Y))) return US_ERR_INVALID_ARG;
    if (split_k < 0 || split_k > W->K / W->TK) return US_ERR_INVALID_ARG;
    const Plan pl = plan_ie(B, N, split_k);
    if (!ws || ws_bytes < pl.ws || !aligned16(ws)) return US_ERR_WORKSPACE;
    UsKParams p;
    fill_common(p, W, N);
    p.X = Xq; p.s_w = s_w; p.s_x = s_x; p.Yacc = Yacc; p.Y = Y;
    p.split = pl.split; p.tok_block = pl.tok_block;
    p.ie_ra = B->RA; p.ie_ca = B->CA; p.perm = B->perm;
    if (pl.sk) {
        p.nTM = W->M / 64;                                    // 64-row bands of super-tiles
        p.ws = ws;
        return us::launch_w4a4_sk_ie(p, static_cast<cudaStream_t>(stream));
    }
    const int ntb = (N + pl.tok_block - 1) / pl.tok_block;
    p.counters = static_cast<unsigned*>(ws);
    p.ws = static_cast<uint8_t*>(ws) + counters_bytes(p.nTM, ntb);
    return us::launch_spmm_generic(p, US_I4, static_cast<cudaStream_t>(stream));
}

us_status us_colinfo(const us_bitmap* W, uint32_t* colinfo, void* stream) {
    if (!W) return US_ERR_INVALID_ARG;
    us_status s = check_bitmap(W, W->elem, US_ORDER_COL);
    if (s != US_OK) return s;
    if (!colinfo || !aligned16(colinfo)) return US_ERR_INVALID_ARG;
    const int64_t nT = (int64_t)(W->M / W->TM) * (W->K / W->TK);
    return us::launch_colinfo(W->bitmap, W->TM, W->TK, nT, colinfo, static_cast<cudaStream_t>(stream));
}

us_status us_spmspv_f16_ci(const us_bitmap* W, const uint32_t* colinfo, const uint16_t* X, int N, float tau,
                           uint16_t* Y, void* ws, size_t ws_bytes, void* stream) {
    us_status s = check_bitmap(W, US_F16, US_ORDER_COL);
    if (s != US_OK) return s;
    if (N < 1 || !colinfo || !X || !Y || !aligned16(colinfo) || !aligned16(X) || !aligned16(Y) || !(tau >= 0.f))
        return US_ERR_INVALID_ARG;
    if ((int64_t)N * W->K >= ((int64_t)1 << 31) || (int64_t)N * W->M >= ((int64_t)1 << 31)) return US_ERR_TOO_LARGE;
    const Plan pl = plan_spmspv(W, false);
    if (pl.ws && (!ws || ws_bytes < pl.ws || !aligned16(ws))) return US_ERR_WORKSPACE;
    UsKParams p;
    fill_common(p, W, N);
    p.X = X; p.Y = Y; p.tau = tau;
    p.split = pl.split; p.tok_block = 1;
    return us::launch_spmspv_ci(p, colinfo, static_cast<cudaStream_t>(stream));
}

us_status us_quantize_x(const uint16_t* X, int N, int K, uint8_t* Xq, uint16_t* s_x, void* stream) {
    if (N < 1 || K < 32 || K % 32 || (int64_t)N * K >= ((int64_t)1 << 32)) return US_ERR_INVALID_ARG;
    if (!X || !Xq || !s_x || !aligned16(X) || !aligned16(Xq)) return US_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(s_x) & 1u) != 0) return US_ERR_INVALID_ARG;
    return us::launch_quantize_x(X, N, K, Xq, s_x, static_cast<cudaStream_t>(stream));
}

us_status us_validate(const us_bitmap* W) {
    if (!W) return US_ERR_INVALID_ARG;
    us_status s = check_shape(W->M, W->K, W->TM, W->TK, W->elem);
    if (s != US_OK) return s;
    if (W->order != US_ORDER_ROW && W->order != US_ORDER_COL) return US_ERR_INVALID_ARG;
    if (!W->bitmap || !W->tile_off || (!W->values && W->values_bytes)) return US_ERR_INVALID_ARG;
    const int nTM = W->M / W->TM, nTK = W->K / W->TK;
    const int64_t nT = (int64_t)nTM * nTK;
    const int64_t wpt = (int64_t)W->TM * W->TK / 64;
    const int bits = W->elem == US_F16 ? 16 : (W->elem == US_I4 ? 4 : 2);
    const uint32_t E = 128u / (uint32_t)bits;
    const uint8_t* vals = static_cast<const uint8_t*>(W->values);
    if (W->tile_off[0] != 0) return US_ERR_CORRUPT;
    for (int64_t t = 0; t < nT; ++t) {
        const uint64_t o0 = W->tile_off[t], o1 = W->tile_off[t + 1];
        if (o1 < o0 || (o1 - o0) % E) return US_ERR_CORRUPT;
        if (o1 * bits > (uint64_t)W->values_bytes * 8) return US_ERR_CORRUPT;
        uint64_t P = 0;
        for (int64_t w = 0; w < wpt; ++w) P += (uint64_t)__builtin_popcountll(W->bitmap[t * wpt + w]);
        if (P > o1 - o0 || (o1 - o0) - P >= E) return US_ERR_CORRUPT;
        for (uint64_t e = o0 + P; e < o1; ++e) {   // padding must be zero
            const uint8_t by = vals[e * bits / 8];
            const uint8_t v = bits == 16 ? by
                            : bits == 4 ? (uint8_t)((e & 1) ? (by >> 4) : (by & 15))
                                        : (uint8_t)((by >> (2 * (e & 3))) & 3);
            if (v || (bits == 16 && vals[e * 2 + 1])) return US_ERR_CORRUPT;
        }
    }
    return US_OK;
}

us_status us_selftest_wait_timeout(uint64_t limit_ns, uint64_t* elapsed_ns, void* stream) {
    if (limit_ns < 1000ull || limit_ns > 1000000000ull) return US_ERR_INVALID_ARG;
    if (elapsed_ns && (reinterpret_cast<uintptr_t>(elapsed_ns) & 7u)) return US_ERR_INVALID_ARG;
    unsigned* status = status_ptr();
    if (!status) return US_ERR_CUDA;
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns, elapsed_ns);
    return cudaGetLastError() == cudaSuccess ? US_OK : US_ERR_CUDA;
}

us_status us_get_last_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return US_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_us_status, sizeof(v)) != cudaSuccess) return US_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_us_status, &zero, sizeof(zero)) != cudaSuccess) return US_ERR_CUDA;
    return static_cast<us_status>(v);
}

}  // extern "C"
