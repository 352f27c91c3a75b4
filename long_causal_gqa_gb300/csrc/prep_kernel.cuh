// Q/K prologue as its own pass: per-head RMS normalisation (times a learned
// weight) and/or the rotary position embedding, applied to every row of a
// [heads][T][128] bf16 tensor. The attention kernel applies the same
// transform to its Q tiles in shared memory; K goes through this pass once
// per call (every K tile is read by many units, so transforming it on each
// load would repeat the work), writing the prepared keys the caller keeps.
//
// The step is the fused Q/K normalisation and rotary embedding that the h3.c
// README places before attention ("Profiling and diagnostic paths",
// "Checkpoint layout and media pipeline"):
//   y = x * rsqrt(mean(x^2) + eps) * w                       (if w given)
//   for i < 64: (y_i, y_{i+64}) <- (y_i c - y_{i+64} s, y_{i+64} c + y_i s),
//   c = cos[t][i], s = sin[t][i]                             (if tables given)
// computed in fp32 and rounded to bf16 once.
#pragma once
#include <cstdint>

namespace h3gqa {

constexpr int kPrepThreads = 256;

// One warp per row; lane l holds dims 4l..4l+3, so the rotation partner of
// lane l < 16 is lane l + 16 (dims i and i + 64). y may be x itself (keys
// prepared in place): every lane's loads of a row feed the warp shuffles
// that come before any store of that row, so no lane overwrites a value
// another lane has yet to read.
__global__ void __launch_bounds__(kPrepThreads)
qk_prep_kernel(const uint16_t *x, uint16_t *y, long long n_rows, long long T,
               const uint16_t *__restrict__ w, float eps, const float *__restrict__ cosv,
               const float *__restrict__ sinv)
{
    const int lane = threadIdx.x & 31;
    const long long n_warps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < n_rows;
         r += n_warps) {
        const long long tok = r % T;
        const uint2 v = reinterpret_cast<const uint2 *>(x + r * 128)[lane];
        float f[4] = {__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                      __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u)};
        if (w != nullptr) {
            float ss = f[0] * f[0] + f[1] * f[1] + f[2] * f[2] + f[3] * f[3];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float rs = rsqrtf(ss * (1.0f / 128.0f) + eps);
            const uint2 wv = __ldg(reinterpret_cast<const uint2 *>(w) + lane);
            f[0] *= rs * __uint_as_float(wv.x << 16);
            f[1] *= rs * __uint_as_float(wv.x & 0xFFFF0000u);
            f[2] *= rs * __uint_as_float(wv.y << 16);
            f[3] *= rs * __uint_as_float(wv.y & 0xFFFF0000u);
        }
        if (cosv != nullptr) {
            const int i0 = (4 * lane) & 63;
            const float4 c = __ldg(reinterpret_cast<const float4 *>(cosv + tok * 64 + i0));
            const float4 s = __ldg(reinterpret_cast<const float4 *>(sinv + tok * 64 + i0));
            const float cs[4] = {c.x, c.y, c.z, c.w}, sn[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float other = __shfl_xor_sync(0xffffffffu, f[e], 16);
                f[e] = lane < 16 ? f[e] * cs[e] - other * sn[e] : f[e] * cs[e] + other * sn[e];
            }
        }
        uint2 out;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out.x) : "f"(f[1]), "f"(f[0]));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out.y) : "f"(f[3]), "f"(f[2]));
        reinterpret_cast<uint2 *>(y + r * 128)[lane] = out;
    }
}

}  // namespace h3gqa
