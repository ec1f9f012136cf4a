// us_w4a4.cu -- W4A4 decode kernel for small token counts (filled in below).
#include "us_common.cuh"
#include "us_internal.h"

namespace us {

bool w4a4_fast_supported(int, int, int) { return false; }

size_t w4a4_fast_ws(int M, int TM, int N, int split) {
    (void)N;
    const int nTM = M / TM;
    const size_t counters = ((size_t)nTM * 4 + 255) & ~(size_t)255;
    return split <= 1 ? counters : counters + (size_t)split * M * N * 4;
}

us_status launch_w4a4_fast(const UsKParams&, cudaStream_t) { return US_ERR_UNSUPPORTED; }

}  // namespace us
