// Q6_K GEMV straight from raw GGUF rows: y = W x with W held exactly as the
// file stores it (no repack).  The decode step streams its Q6_K weights from
// the planar layout instead (the GEMV engine); this kernel is the building
// block for a caller that holds the file's bytes.
//
// Q6_K block (256 weights, 210 bytes, "k-quants" super-block format): ql[128]
// low nibbles, qh[64] high bit pairs, int8 scales[16] (one per 16 weights),
// fp16 d.  In half h (128 weights) and column c < 32 the byte pair
// ql[64h + c], ql[64h + 32 + c] and qh[32h + c] give the four 6-bit codes of
// weights 128h + c + 32s (s = 0..3): low nibbles for s = 0, 1, high nibbles
// for s = 2, 3, bit pair 2s of the qh byte on top; weight = d * scales[8h +
// c/16 + 2s] * (code - 32).
//
// One warp per two rows.  A row's bytes go through a shared buffer in
// chunks of up to kChunkBlocks blocks: 210-byte blocks leave a chunk only
// 2-byte aligned, so the 16-byte-aligned middle of its byte range streams in
// by 16-byte async copies (coalesced, no registers held) and the ragged head
// and tail (under 16 bytes each) by 2-byte loads; every access stays inside
// the chunk's own bytes.  Shared offsets keep the global address modulo 16,
// so the async copies land 16-byte aligned, and a lane's eight bytes of a
// block are read with 32- or 64-bit shared loads whatever the block's
// alignment.
#include <cuda_fp16.h>

#include "qg_host.cuh"

namespace qg {
namespace {

constexpr int kQ6Bytes = 210;
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 2;  // every x load serves both rows
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;
constexpr int kChunkBlocks = 16;
// one row's chunk: 16 bytes of front pad (the 32-bit loads of a 2-mod-4 address
// start 2 bytes early), the chunk's offset modulo 16, the chunk, and 16 bytes
// of back pad (they end up to 2 bytes late)
constexpr int kRowBuf = 16 + 16 + kChunkBlocks * kQ6Bytes + 16;  // 3408, a multiple of 16
constexpr int kRowsSmem = kRowsPerCta * kRowBuf;
static_assert(kRowBuf % 16 == 0, "per-row buffers must stay 16-byte aligned");

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Bytes q[0..7] of a shared buffer as two words, q 2-byte aligned.  The
// address modulo 8 is the same for every lane of a warp here (a block's
// start plus multiples of 8), so the branch is uniform: one 64-bit load, two
// 32-bit loads, or three 32-bit loads from 2 bytes early joined by funnel
// shifts.
__device__ __forceinline__ uint2 ld8(const uint8_t* q) {
    const unsigned r = static_cast<unsigned>(reinterpret_cast<uintptr_t>(q)) & 7u;
    if (r == 0) return *reinterpret_cast<const uint2*>(q);
    if (r == 4) return make_uint2(*reinterpret_cast<const unsigned*>(q), *reinterpret_cast<const unsigned*>(q + 4));
    const unsigned* w = reinterpret_cast<const unsigned*>(q - 2);
    const unsigned w0 = w[0], w1 = w[1], w2 = w[2];
    return make_uint2(__funnelshift_r(w0, w1, 16), __funnelshift_r(w1, w2, 16));
}

// Lane l = 16 h + 4 g + 2 i + e takes half h, 32-weight group g, and the
// eight columns c = 16 i + 8 e .. c + 7 of that group: one 16-weight
// sub-block's half, so one scale, sc[8h + i + 2g].  Its weights are
// 128 h + 32 g + c + j.  A 6-bit code becomes an exact float by the mantissa
// of 2^23: the word 0x4B000000 | code is 2^23 + code, and subtracting 2^23 + 32
// leaves code - 32 (a byte permute and an add; no integer conversion).  With
// d * sc exact in f32 (11 x 8 bits), a lane's block sum is
// fma(d * sc, sum_j (code_j - 32) x_j, acc).
__device__ __forceinline__ float code_f(unsigned codes, unsigned sel) {
    return __int_as_float(static_cast<int>(__byte_perm(codes, 0x4B000000u, sel))) - 8388640.0f;  // 2^23 + 32
}
__device__ __forceinline__ float block_dot(const uint8_t* blk, const float4& xa, const float4& xc, float acc, int h,
                                           int g, int i, int c) {
    const uint2 ql = ld8(blk + 64 * h + 32 * (g & 1) + c);
    const uint2 qh = ld8(blk + 128 + 32 * h + c);
    const unsigned sh = 4u * static_cast<unsigned>(g >> 1), hs = 2u * static_cast<unsigned>(g);
    const unsigned c0 = ((ql.x >> sh) & 0x0F0F0F0Fu) | (((qh.x >> hs) & 0x03030303u) << 4);
    const unsigned c1 = ((ql.y >> sh) & 0x0F0F0F0Fu) | (((qh.y >> hs) & 0x03030303u) << 4);
    const unsigned sc_u8 = blk[192 + 8 * h + i + 2 * g];
    const float scf = __int_as_float(static_cast<int>(0x4B000000u | (sc_u8 ^ 0x80u))) - 8388736.0f;  // 2^23 + 128
    const float d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
    float t = code_f(c0, 0x7540u) * xa.x;
    t = fmaf(code_f(c0, 0x7541u), xa.y, t);
    t = fmaf(code_f(c0, 0x7542u), xa.z, t);
    t = fmaf(code_f(c0, 0x7543u), xa.w, t);
    t = fmaf(code_f(c1, 0x7540u), xc.x, t);
    t = fmaf(code_f(c1, 0x7541u), xc.y, t);
    t = fmaf(code_f(c1, 0x7542u), xc.z, t);
    t = fmaf(code_f(c1, 0x7543u), xc.w, t);
    return fmaf(d * scf, t, acc);
}

// Issue the copies of blocks [c0, c0 + cb) of one row into buf; returns the
// shared address of the chunk's first block.
__device__ __forceinline__ const uint8_t* stage_chunk(const uint8_t* w, int row, int nb, int c0, int cb, uint8_t* buf,
                                                      int lane) {
    constexpr uintptr_t kLow = 15;
    const uintptr_t S = reinterpret_cast<uintptr_t>(w) + (static_cast<size_t>(row) * nb + c0) * kQ6Bytes;
    const uintptr_t E = S + static_cast<uintptr_t>(cb) * kQ6Bytes;
    const uintptr_t base = S & ~kLow;  // address p sits at data + (p - base)
    const uintptr_t A = min((S + kLow) & ~kLow, E);
    const uintptr_t B = max(E & ~kLow, A);
    uint8_t* data = buf + 16;
    // [S, A) and [B, E): under 16 bytes each, 2-byte loads; [A, B): 16-byte async copies
    const int nhead = static_cast<int>((A - S) >> 1), ntail = static_cast<int>((E - B) >> 1);
    const int nvec = static_cast<int>((B - A) >> 4);
    for (int v = lane; v < nvec; v += 32)
        cp_async16(data + (A - base) + 16 * v, reinterpret_cast<const void*>(A + 16 * static_cast<uintptr_t>(v)));
    if (lane < nhead)
        *reinterpret_cast<uint16_t*>(data + (S - base) + 2 * lane) =
            __ldg(reinterpret_cast<const uint16_t*>(S + 2 * static_cast<uintptr_t>(lane)));
    else if (lane >= 16 && lane - 16 < ntail)
        *reinterpret_cast<uint16_t*>(data + (B - base) + 2 * (lane - 16)) =
            __ldg(reinterpret_cast<const uint16_t*>(B + 2 * static_cast<uintptr_t>(lane - 16)));
    return data + (S - base);
}

__global__ void __launch_bounds__(32 * kWarps) q6k_rows_kernel(const uint8_t* __restrict__ w,
                                                               const float* __restrict__ x,
                                                               float* __restrict__ y, int n, int nb) {
    extern __shared__ __align__(16) uint8_t rows_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * kWarps + warp) * kRowsPerWarp;
    if (row0 >= n) return;  // the warps of a CTA never synchronise with one another
    const int nr = min(kRowsPerWarp, n - row0);
    uint8_t* buf = rows_smem + warp * kRowsPerWarp * kRowBuf;
    const int h = lane >> 4, g = (lane >> 2) & 3, i = (lane >> 1) & 1, c = 16 * i + 8 * (lane & 1);
    float acc[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) acc[r] = 0.f;
    for (int c0 = 0; c0 < nb; c0 += kChunkBlocks) {
        const int cb = min(kChunkBlocks, nb - c0);
        const uint8_t* blk[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
            blk[r] = r < nr ? stage_chunk(w, row0 + r, nb, c0, cb, buf + r * kRowBuf, lane) : nullptr;
        cp_async_wait_all();
        __syncwarp();
        const float* xb = x + 256 * c0 + 128 * h + 32 * g + c;
        for (int b = 0; b < cb; ++b, xb += 256) {
            const float4 xa = __ldg(reinterpret_cast<const float4*>(xb));
            const float4 xc = __ldg(reinterpret_cast<const float4*>(xb + 4));
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r)
                if (r < nr) acc[r] = block_dot(blk[r] + b * kQ6Bytes, xa, xc, acc[r], h, g, i, c);
        }
        __syncwarp();  // every lane is done with the buffers before the next chunk overwrites them
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        float a = acc[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0 && r < nr) y[row0 + r] = a;
    }
}

}  // namespace
}  // namespace qg

using namespace qg;

extern "C" int qg_gemv_q6k(const void* w, const float* x, float* y, int n, int k, qg_stream stream) {
    if (!w || !x || !y) return set_err(QG_ERR_ARG, "gemv_q6k: NULL pointer");
    if (n < 0 || k < 0) return set_err(QG_ERR_ARG, "gemv_q6k: negative size n=%d k=%d", n, k);
    if (n == 0 || k == 0) return set_err(QG_ERR_EMPTY, "gemv_q6k: empty tensor n=%d k=%d", n, k);
    if (k % 256) return set_err(QG_ERR_SHAPE, "gemv_q6k: k=%d is not a multiple of 256", k);
    if ((reinterpret_cast<uintptr_t>(w) & 1u) || (reinterpret_cast<uintptr_t>(x) & 15u) ||
        (reinterpret_cast<uintptr_t>(y) & 3u))
        return set_err(QG_ERR_ARG, "gemv_q6k: w must be 2-byte, x 16-byte and y 4-byte aligned");
    const int rc = grant_smem(reinterpret_cast<const void*>(q6k_rows_kernel), kRowsSmem);
    if (rc) return rc;
    const unsigned grid = static_cast<unsigned>((n + kRowsPerCta - 1) / kRowsPerCta);
    q6k_rows_kernel<<<grid, 32 * kWarps, kRowsSmem, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(w), x, y, n, k / 256);
    QG_CUDA(cudaGetLastError());
    return QG_OK;
}
