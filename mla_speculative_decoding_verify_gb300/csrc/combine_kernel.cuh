// Log-sum-exp merge of split-KV partials (flash-decoding combine).  One warp
// per output row; each lane owns 16 of the 512 columns.  Memory-bound: it
// reads num_splits * 2 KB + num_splits * 4 B per row and writes 2 KB + 4 B.
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace mla {

constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32)
mla_combine_kernel(const float* __restrict__ part_out, const float* __restrict__ part_lse, int num_splits,
                   long long rows, float* __restrict__ out, float* __restrict__ lse) {
    grid_dependency_wait();     // the verify kernel's partials
    const int lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    // max over the splits' lse (natural log)
    float m = -INFINITY;
    for (int s = lane; s < num_splits; s += 32) m = fmaxf(m, part_lse[static_cast<long long>(s) * rows + row]);
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float4 acc[4];
    for (int u = 0; u < 4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m == -INFINITY) {
        float4* dst = reinterpret_cast<float4*>(out + row * 512);
        for (int u = 0; u < 4; ++u) dst[lane + 32 * u] = acc[u];
        if (lane == 0) lse[row] = -INFINITY;
        return;
    }
    float z = 0.f;
    for (int s = lane; s < num_splits; s += 32) z += __expf(part_lse[static_cast<long long>(s) * rows + row] - m);
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float lse_row = m + __logf(z);
    for (int s = 0; s < num_splits; ++s) {
        const float ls = part_lse[static_cast<long long>(s) * rows + row];
        const float w = (ls == -INFINITY) ? 0.f : __expf(ls - lse_row);
        const float4* src = reinterpret_cast<const float4*>(part_out + (static_cast<long long>(s) * rows + row) * 512);
        for (int u = 0; u < 4; ++u) {
            const float4 v = __ldg(src + lane + 32 * u);
            acc[u].x += w * v.x;
            acc[u].y += w * v.y;
            acc[u].z += w * v.z;
            acc[u].w += w * v.w;
        }
    }
    float4* dst = reinterpret_cast<float4*>(out + row * 512);
    for (int u = 0; u < 4; ++u) dst[lane + 32 * u] = acc[u];
    if (lane == 0) lse[row] = lse_row;
}

}  // namespace mla
