// Launch order of the kernels that walk one (sequence, head) unit's chunks
// per CTA (the scan kernels, the CUDA-core forward, the backward's reverse
// walk).
#pragma once

#include <climits>

#include "dn_internal.h"

namespace dn {

// With offsets (sequences of different lengths) a kernel that walks each
// (sequence, head) unit's chunks in one CTA takes its units longest sequence
// first: when the CTAs outnumber the SMs, the block scheduler hands the later
// ones to SMs as earlier ones finish, and starting the longest walks first
// shortens the launch (a longest-processing-time order).  The sequence of
// rank r (the CTA's unit index over the units of one sequence), ties going by
// index; up to kSortSeqs sequences, else the rank is the sequence.  Every
// lane of the calling warp takes part; each warp works it out for itself.
constexpr int kSortSeqs = 64;
__device__ __forceinline__ int seq_of_rank(const Params &p, int r, int lane) {
    if (!p.cu || p.N <= 1 || p.N > kSortSeqs) return r;
    auto len = [&](int m) -> int {
        const long long l = m < p.N ? p.cu[m + 1] - p.cu[m] : -1;
        return (int)max(min(l, (long long)INT_MAX), (long long)-1);
    };
    const int la = len(lane), lb = len(lane + 32);
    int ra = 0, rb = 0;  // ranks of sequences lane and lane + 32
    for (int j = 0; j < p.N; ++j) {
        const int lj = __shfl_sync(0xffffffffu, j < 32 ? la : lb, j & 31);
        ra += (lj > la) || (lj == la && j < lane);
        rb += (lj > lb) || (lj == lb && j < lane + 32);
    }
    int n = -1;
    if (lane < p.N && ra == r) n = lane;
    if (lane + 32 < p.N && rb == r) n = lane + 32;
    return __reduce_max_sync(0xffffffffu, n);
}

}  // namespace dn
