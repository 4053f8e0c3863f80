// Q6_K GEMV straight from raw GGUF rows: y = W x with W held exactly as the
// file stores it (no repack), one warp per row.  The decode step streams its
// Q6_K weights from the planar layout instead (the GEMV engine); this kernel
// is the building block for a caller that holds the file's bytes.
//
// Q6_K block (256 weights, 210 bytes, "k-quants" super-block format): ql[128]
// low nibbles, qh[64] high bit pairs, int8 scales[16] (one per 16 weights),
// fp16 d.  In half h (128 weights) and column c < 32 the byte pair
// ql[64h + c], ql[64h + 32 + c] and qh[32h + c] give the four 6-bit codes of
// weights 128h + c + 32s (s = 0..3): low nibbles for s = 0, 1, high nibbles
// for s = 2, 3, bit pair 2s of the qh byte on top; weight = d * scales[8h +
// c/16 + 2s] * (code - 32).
#include <cuda_fp16.h>

#include "qg_host.cuh"

namespace qg {
namespace {

constexpr int kQ6Bytes = 210;
constexpr int kRowsPerCta = 8;  // one warp per row

// Lane l of a row's warp takes half h = l / 16 and the column pair
// c = 2 (l % 16), c + 1 of every block: eight weights, two per scale.
__global__ void __launch_bounds__(32 * kRowsPerCta) q6k_rows_kernel(const uint8_t* __restrict__ w,
                                                                    const float* __restrict__ x,
                                                                    float* __restrict__ y, int n, int nb) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
    if (row >= n) return;
    const int h = lane >> 4, c = 2 * (lane & 15), is = c >> 4;
    const uint8_t* blk = w + static_cast<size_t>(row) * nb * kQ6Bytes;
    const float* xb = x + 128 * h + c;
    float acc = 0.f;
#pragma unroll 4
    for (int b = 0; b < nb; ++b, blk += kQ6Bytes, xb += 256) {
        const unsigned lo = __ldg(reinterpret_cast<const uint16_t*>(blk + 64 * h + c));
        const unsigned hi = __ldg(reinterpret_cast<const uint16_t*>(blk + 64 * h + 32 + c));
        const unsigned qh = __ldg(reinterpret_cast<const uint16_t*>(blk + 128 + 32 * h + c));
        const int8_t* sc = reinterpret_cast<const int8_t*>(blk + 192 + 8 * h + is);
        const float d = __half2float(__ldg(reinterpret_cast<const __half*>(blk + 208)));
        float s = 0.f;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            // the nibble source: low nibbles of ql[c..] for g = 0, of ql[32 + c..]
            // for g = 1, their high nibbles for g = 2, 3
            const unsigned src = (g & 1) ? hi : lo, sh = (g >> 1) * 4;
            const int q0 = static_cast<int>(((src >> sh) & 15u) | (((qh >> (2 * g)) & 3u) << 4)) - 32;
            const int q1 = static_cast<int>(((src >> (8 + sh)) & 15u) | (((qh >> (8 + 2 * g)) & 3u) << 4)) - 32;
            const float2 xv = __ldg(reinterpret_cast<const float2*>(xb + 32 * g));
            const float t = fmaf(static_cast<float>(q1), xv.y, static_cast<float>(q0) * xv.x);
            s = fmaf(static_cast<float>(__ldg(sc + 2 * g)), t, s);
        }
        acc = fmaf(d, s, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) y[row] = acc;
}

}  // namespace
}  // namespace qg

using namespace qg;

extern "C" int qg_gemv_q6k(const void* w, const float* x, float* y, int n, int k, qg_stream stream) {
    if (!w || !x || !y) return set_err(QG_ERR_ARG, "gemv_q6k: NULL pointer");
    if (n < 0 || k < 0) return set_err(QG_ERR_ARG, "gemv_q6k: negative size n=%d k=%d", n, k);
    if (n == 0 || k == 0) return set_err(QG_ERR_EMPTY, "gemv_q6k: empty tensor n=%d k=%d", n, k);
    if (k % 256) return set_err(QG_ERR_SHAPE, "gemv_q6k: k=%d is not a multiple of 256", k);
    if ((reinterpret_cast<uintptr_t>(w) & 1u) || (reinterpret_cast<uintptr_t>(x) & 7u) ||
        (reinterpret_cast<uintptr_t>(y) & 3u))
        return set_err(QG_ERR_ARG, "gemv_q6k: w must be 2-byte, x 8-byte and y 4-byte aligned");
    const unsigned grid = static_cast<unsigned>((n + kRowsPerCta - 1) / kRowsPerCta);
    q6k_rows_kernel<<<grid, 32 * kRowsPerCta, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(w), x, y, n, k / 256);
    QG_CUDA(cudaGetLastError());
    return QG_OK;
}
