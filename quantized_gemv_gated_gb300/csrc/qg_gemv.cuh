// GEMV engine for GGUF k-quant weights on GB300 (sm_103a).
//
// y[n] = sum_k deq(W[n][k]) * x[k], one launch per projection (or per group
// of projections sharing an input), in the role of the float ("mwv") Q4_K /
// Q6_K GEMV of forward_qwen35_cuda.rs (gemv_dispatch, pin_float_gemv).
//
// Memory side.  Each CTA owns a contiguous range of rows (in units of 8).  A
// producer warp streams them global -> shared with 1-D bulk copies
// (cp.async.bulk, the TMA engine) into a ring of stages guarded by mbarriers,
// with an L2 evict-first policy (weights are read once per token).  The copies
// are issued at kernel start, before the programmatic-dependent-launch wait,
// so a kernel's weights stream in while the previous kernel finishes.
//
// Arithmetic side.  x (K floats, after the kernel's prologue: RMSNorm, gated
// norm, ...) is held in shared memory as a 24-bit block-fixed-point integer
// per element: in every 256-element block (one k-quant super-block of the
// weights), n_i = rint(x_i * 2^(22-e)) with 2^e <= max|x| < 2^(e+1), so
// |n_i| < 2^23 and the representation keeps the 24 significant bits of the
// block's largest element (f32 keeps 24).  n_i is stored as three byte planes
// (n = n2*65536 + n1*256 + n0, n2 signed), every sum of quant*n over a
// sub-block is computed EXACTLY with dp4a integer dot products, and the
// sub-block sums of a 64-weight chunk are weighted by their integer scales in
// integer arithmetic; one float per chunk is accumulated in f32.  This is not
// the int8 activation quantisation forward_qwen35_cuda.rs rejects
// (pin_float_gemv): the only rounding of x is below 2^-23 of its block's
// largest magnitude, and the integer sums carry no rounding at all.
//
//   Q4_K sub-block j (32 weights): d*sc_j*sum(q*x) - dmin*m_j*sum(x)
//   Q6_K group of 16 weights:      d*sc*sum((q-32)*x)
#pragma once
#include "qg_common.cuh"

namespace qg {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxStages = 8;
constexpr int QT_Q4K = 12;
constexpr int QT_Q6K = 14;

// Geometry of one launch (identical on host and device).
struct GemvShape {
    const uint8_t* w0;  // Q4_K: GGUF rows; Q6_K: planar base
    const uint8_t* w1;  // second matrix of a dual launch (same shape), else null
    int n, n8, k, nb, cr;
    int lg;      // log2(lanes per row)
    int rs;      // rows per stage (multiple of 8 * rows per warp)
    int stages;  // ring depth
    int units;   // ceil(n / 8)
    int stage_bytes;
    int pro_floats;  // prologue scratch floats
    int rows_cta;    // most rows one CTA owns (row-result buffer of deferred epilogues)
    unsigned* err;
    L2Prefetch next;  // operands of the next kernel, pulled into L2 by the producer
};

// Shared-memory layout offsets.  aux: per 256-element super-block the unit
// 2^(e-22) (float), then Q4_K: per 32-element sub-block the sum of n (float);
// Q6_K: per 16-element group {-32*N0, -32*N1, -32*N2, 0} (digit-plane sums).
__host__ __device__ inline int xaux_bytes(int qt, int k) {
    return ((4 * (k / 256) + 15) & ~15) + (qt == QT_Q4K ? 4 * (k / 32) : k);
}
__host__ __device__ inline int aux_tail(int k) { return (4 * (k / 256) + 15) & ~15; }
__host__ __device__ inline int off_dig() { return 16 * kMaxStages; }
__host__ __device__ inline int off_aux(int k) { return off_dig() + 3 * k; }
__host__ __device__ inline int off_pro(int qt, int k) { return ((off_aux(k) + xaux_bytes(qt, k)) + 15) & ~15; }
__host__ __device__ inline int off_ys(int qt, int k, int pro_floats) { return off_pro(qt, k) + 4 * pro_floats; }
__host__ __device__ inline int off_ring(int qt, int k, int pro_floats, int ys_floats) {
    return (off_ys(qt, k, pro_floats) + 4 * ys_floats + 127) & ~127;
}

// 16-byte-unit swizzles of the digit planes, chosen so that the 8 lanes of
// one shared-memory phase read 8 distinct bank groups.
__device__ __forceinline__ unsigned swz(int qt, unsigned u) {
    return qt == QT_Q4K ? (u ^ ((u >> 3) & 3u)) : (u ^ ((u >> 2) & 6u));
}

__device__ __forceinline__ unsigned dp4a_uu(unsigned a, unsigned b, unsigned c) { return __dp4a(a, b, c); }
__device__ __forceinline__ int dp4a_us(unsigned a, unsigned b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(unsigned a, unsigned b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---------------------------------------------------------- x representation
// One warp per 256-element super-block, 8 consecutive elements per lane:
// n_i = rint(x_i * 2^(22-e)) with 2^e <= max|x| over the super-block
// (clamped to |n| < 2^23), stored as three byte planes.
template <int QT, class Pro>
__device__ void build_xrep(const Pro& pro, const float* sm, uint8_t* dig, uint8_t* aux, int k, int warp,
                           int lane) {
    const int nsb = k >> 8;
    float* units = reinterpret_cast<float*>(aux);
    for (int b = warp; b < nsb; b += kConsumerWarps) {
        const int i0 = 256 * b + 8 * lane;
        float x[8];
        unsigned am = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            x[j] = pro.value(sm, i0 + j);
            am = max(am, __float_as_uint(x[j]) & 0x7fffffffu);
        }
        am = __reduce_max_sync(FULL, am);
        int e = static_cast<int>(am >> 23) - 127;
        e = e < -100 ? -100 : e;
        const float mul = __uint_as_float(static_cast<unsigned>(149 - e) << 23);   // 2^(22-e)
        const float unit = __uint_as_float(static_cast<unsigned>(105 + e) << 23);  // 2^(e-22)
        unsigned w0[2] = {0u, 0u}, w1[2] = {0u, 0u}, w2[2] = {0u, 0u};
        int nsum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int n = __float2int_rn(x[j] * mul);
            n = n > 8388607 ? 8388607 : (n < -8388607 ? -8388607 : n);
            nsum += n;
            const int sh = 8 * (j & 3);
            w0[j >> 2] |= static_cast<unsigned>(n & 255) << sh;
            w1[j >> 2] |= static_cast<unsigned>((n >> 8) & 255) << sh;
            w2[j >> 2] |= static_cast<unsigned>((n >> 16) & 255) << sh;
        }
        const unsigned u = static_cast<unsigned>(i0) >> 4;
        const unsigned off = (swz(QT, u) << 4) + 8 * (lane & 1);
        *reinterpret_cast<uint2*>(dig + off) = make_uint2(w0[0], w0[1]);
        *reinterpret_cast<uint2*>(dig + k + off) = make_uint2(w1[0], w1[1]);
        *reinterpret_cast<uint2*>(dig + 2 * k + off) = make_uint2(w2[0], w2[1]);
        if (lane == 0) units[b] = unit;
        if constexpr (QT == QT_Q4K) {
            nsum += __shfl_xor_sync(FULL, nsum, 1);
            nsum += __shfl_xor_sync(FULL, nsum, 2);
            if ((lane & 3) == 0)
                reinterpret_cast<float*>(aux + aux_tail(k))[8 * b + (lane >> 2)] = static_cast<float>(nsum);
        } else {
            int n0 = static_cast<int>(dp4a_uu(w0[0], 0x01010101u, dp4a_uu(w0[1], 0x01010101u, 0u)));
            int n1 = static_cast<int>(dp4a_uu(w1[0], 0x01010101u, dp4a_uu(w1[1], 0x01010101u, 0u)));
            int n2 = dp4a_su(w2[0], 0x01010101u, dp4a_su(w2[1], 0x01010101u, 0));
            n0 += __shfl_xor_sync(FULL, n0, 1);
            n1 += __shfl_xor_sync(FULL, n1, 1);
            n2 += __shfl_xor_sync(FULL, n2, 1);
            if ((lane & 1) == 0)
                reinterpret_cast<int4*>(aux + aux_tail(k))[swz(QT, u)] = make_int4(-32 * n0, -32 * n1, -32 * n2, 0);
        }
    }
}

// ------------------------------------------------------------ chunk kernels
// One lane, one 64-weight chunk.  Sub-block sums are exact integers; they are
// weighted by their integer scales in integer arithmetic and turned into one
// float per chunk, scaled by the super-block's unit.
// Q4_K: group g (sub-blocks 2g and 2g+1) of super-block `blk`, x offset xo.
__device__ __forceinline__ void chunk_q4k(const uint8_t* blk, int g, int xo, const uint8_t* dig,
                                          const uint8_t* aux, int k, float& acc) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 16 + 32 * g);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 32 + 32 * g);
    const unsigned u0 = static_cast<unsigned>(xo) >> 4;
    unsigned a0 = 0, a1 = 0, b0 = 0, b1 = 0;
    int a2 = 0, b2 = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint4 q = h ? qb : qa;
        const unsigned ul = swz(QT_Q4K, u0 + h) << 4, uh = swz(QT_Q4K, u0 + 2 + h) << 4;
        const uint4 l0 = *reinterpret_cast<const uint4*>(dig + ul);
        const uint4 l1 = *reinterpret_cast<const uint4*>(dig + k + ul);
        const uint4 l2 = *reinterpret_cast<const uint4*>(dig + 2 * k + ul);
        const uint4 h0 = *reinterpret_cast<const uint4*>(dig + uh);
        const uint4 h1 = *reinterpret_cast<const uint4*>(dig + k + uh);
        const uint4 h2 = *reinterpret_cast<const uint4*>(dig + 2 * k + uh);
        const unsigned qw[4] = {q.x, q.y, q.z, q.w};
        const unsigned L0[4] = {l0.x, l0.y, l0.z, l0.w}, L1[4] = {l1.x, l1.y, l1.z, l1.w},
                       L2[4] = {l2.x, l2.y, l2.z, l2.w};
        const unsigned H0[4] = {h0.x, h0.y, h0.z, h0.w}, H1[4] = {h1.x, h1.y, h1.z, h1.w},
                       H2[4] = {h2.x, h2.y, h2.z, h2.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const unsigned lo = qw[w] & 0x0f0f0f0fu, hi = (qw[w] >> 4) & 0x0f0f0f0fu;
            a0 = dp4a_uu(lo, L0[w], a0);
            a1 = dp4a_uu(lo, L1[w], a1);
            a2 = dp4a_us(lo, L2[w], a2);
            b0 = dp4a_uu(hi, H0[w], b0);
            b1 = dp4a_uu(hi, H1[w], b1);
            b2 = dp4a_us(hi, H2[w], b2);
        }
    }
    // scale / min of sub-blocks j = 2g (low nibbles) and 2g+1 (high nibbles)
    const float d = f16_to_f32(static_cast<uint16_t>(hdr.x & 0xffffu));
    const float dmin = f16_to_f32(static_cast<uint16_t>(hdr.x >> 16));
    int sc[2], mn[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int j = 2 * g + t, sh = 8 * (j & 3);
        const unsigned by = (hdr.y >> sh) & 0xffu, bz = (hdr.z >> sh) & 0xffu, bw = (hdr.w >> sh) & 0xffu;
        if (j < 4) {
            sc[t] = static_cast<int>(by & 63u);
            mn[t] = static_cast<int>(bz & 63u);
        } else {
            sc[t] = static_cast<int>((bw & 15u) | ((by >> 6) << 4));
            mn[t] = static_cast<int>((bw >> 4) | ((bz >> 6) << 4));
        }
    }
    // |sc * sum| < 63 * 15 * 255 * 32 per sub-block: the weighted sums fit in int32
    const int I0 = sc[0] * static_cast<int>(a0) + sc[1] * static_cast<int>(b0);
    const int I1 = sc[0] * static_cast<int>(a1) + sc[1] * static_cast<int>(b1);
    const int I2 = sc[0] * a2 + sc[1] * b2;
    const float F = fmaf(static_cast<float>(I2), 65536.0f, fmaf(static_cast<float>(I1), 256.0f, static_cast<float>(I0)));
    const float2 ns = *reinterpret_cast<const float2*>(aux + aux_tail(k) + 4 * (xo >> 5));
    const float M = fmaf(static_cast<float>(mn[0]), ns.x, static_cast<float>(mn[1]) * ns.y);
    const float unit = reinterpret_cast<const float*>(aux)[xo >> 8];
    acc = fmaf(unit, fmaf(d, F, -(dmin * M)), acc);
}

// Q6_K planar: quarter-chunk cq = 2*half + part of super-block b (x offset 256*b).
__device__ __forceinline__ void chunk_q6k(const uint8_t* ql, const uint8_t* qhp, const uint8_t* scp,
                                          const uint16_t* dp, int b, int cq, const uint8_t* dig,
                                          const uint8_t* aux, int k, float& acc) {
    const int half = cq >> 1, part = cq & 1;
    const int f = b & 1;  // read the two 16-byte pieces in an order that avoids bank conflicts
    const uint4 p0 = *reinterpret_cast<const uint4*>(ql + 32 * cq + 16 * f);
    const uint4 p1 = *reinterpret_cast<const uint4*>(ql + 32 * cq + 16 * (1 - f));
    const uint4 A = f ? p1 : p0;  // ql[64*half + 16*part ..]      quarters 0 (low), 2 (high)
    const uint4 B = f ? p0 : p1;  // ql[64*half + 32 + 16*part ..] quarters 1 (low), 3 (high)
    const uint4 H = *reinterpret_cast<const uint4*>(qhp + 16 * cq);
    const uint2 S = *reinterpret_cast<const uint2*>(scp + 8 * half);
    const float d = f16_to_f32(*dp);
    const unsigned Aw[4] = {A.x, A.y, A.z, A.w}, Bw[4] = {B.x, B.y, B.z, B.w}, Hw[4] = {H.x, H.y, H.z, H.w};
    const int4* gc = reinterpret_cast<const int4*>(aux + aux_tail(k));
    int I0 = 0, I1 = 0, I2 = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int pos = 256 * b + 128 * half + 32 * s + 16 * part;
        const unsigned u = swz(QT_Q6K, static_cast<unsigned>(pos) >> 4);
        const int4 gcv = gc[u];
        const uint4 D0 = *reinterpret_cast<const uint4*>(dig + (u << 4));
        const uint4 D1 = *reinterpret_cast<const uint4*>(dig + k + (u << 4));
        const uint4 D2 = *reinterpret_cast<const uint4*>(dig + 2 * k + (u << 4));
        const unsigned d0[4] = {D0.x, D0.y, D0.z, D0.w}, d1[4] = {D1.x, D1.y, D1.z, D1.w},
                       d2[4] = {D2.x, D2.y, D2.z, D2.w};
        int t0 = gcv.x, t1 = gcv.y, t2 = gcv.z;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            unsigned q;
            if (s == 0) q = (Aw[w] & 0x0f0f0f0fu) | ((Hw[w] << 4) & 0x30303030u);
            else if (s == 1) q = (Bw[w] & 0x0f0f0f0fu) | ((Hw[w] << 2) & 0x30303030u);
            else if (s == 2) q = ((Aw[w] >> 4) & 0x0f0f0f0fu) | (Hw[w] & 0x30303030u);
            else q = ((Bw[w] >> 4) & 0x0f0f0f0fu) | ((Hw[w] >> 2) & 0x30303030u);
            t0 = static_cast<int>(dp4a_uu(q, d0[w], static_cast<unsigned>(t0)));
            t1 = static_cast<int>(dp4a_uu(q, d1[w], static_cast<unsigned>(t1)));
            t2 = dp4a_us(q, d2[w], t2);
        }
        const int si = part + 2 * s;
        const int sc = static_cast<int>(static_cast<int8_t>(((si < 4 ? S.x : S.y) >> (8 * (si & 3))) & 0xffu));
        // |sc * t| <= 128 * 32 * 255 * 16 per group, four groups: fits in int32
        I0 += sc * t0;
        I1 += sc * t1;
        I2 += sc * t2;
    }
    const float F = fmaf(static_cast<float>(I2), 65536.0f, fmaf(static_cast<float>(I1), 256.0f, static_cast<float>(I0)));
    acc = fmaf(d * reinterpret_cast<const float*>(aux)[b], F, acc);
}

// Partial dot product of one row over the chunks c = lg0, lg0 + G, ...
template <int QT>
__device__ __forceinline__ float row_partial(const uint8_t* stage, int rs, int lrow, int nb, int cr, int G, int lg0,
                                             const uint8_t* dig, const uint8_t* aux, int k) {
    float acc = 0.0f;
    if constexpr (QT == QT_Q4K) {
        const uint8_t* row = stage + static_cast<size_t>(lrow) * nb * 144;
        for (int c = lg0; c < cr; c += G) chunk_q4k(row + (c >> 2) * 144, c & 3, 64 * c, dig, aux, k, acc);
    } else {
        const uint8_t* ql = stage + static_cast<size_t>(lrow) * nb * 128;
        const uint8_t* qh = stage + static_cast<size_t>(rs) * nb * 128 + static_cast<size_t>(lrow) * nb * 64;
        const uint8_t* sc = stage + static_cast<size_t>(rs) * nb * 192 + static_cast<size_t>(lrow) * nb * 16;
        const uint16_t* dd =
            reinterpret_cast<const uint16_t*>(stage + static_cast<size_t>(rs) * nb * 208) + static_cast<size_t>(lrow) * nb;
        for (int c = lg0; c < cr; c += G) {
            const int b = c >> 2;
            chunk_q6k(ql + b * 128, qh + b * 64, sc + b * 16, dd + b, b, c & 3, dig, aux, k, acc);
        }
    }
    return acc;
}

// The chunks c in [4 b0, 4 (b0 + kbs)) with c == lg0 (mod G) of one row,
// accumulated into acc in chunk order, from a stage holding ur rows x kbs
// super-blocks that start at block b0 (Q6_K: its D region holds whole rows of
// nb blocks).  A row split over consecutive stages sums exactly as in one.
template <int QT>
__device__ __forceinline__ float row_acc_slice(const uint8_t* stage, int ur, int lrow, int kbs, int b0, int nb, int G,
                                               int lg0, const uint8_t* dig, const uint8_t* aux, int k, float acc) {
    const int c_lo = 4 * b0, c_hi = 4 * (b0 + kbs);
    int c = c_lo + ((lg0 - c_lo) & (G - 1));
    if constexpr (QT == QT_Q4K) {
        const uint8_t* row = stage + static_cast<size_t>(lrow) * kbs * 144;
        for (; c < c_hi; c += G) chunk_q4k(row + ((c >> 2) - b0) * 144, c & 3, 64 * c, dig, aux, k, acc);
    } else {
        const uint8_t* ql = stage + static_cast<size_t>(lrow) * kbs * 128;
        const uint8_t* qh = stage + static_cast<size_t>(ur) * kbs * 128 + static_cast<size_t>(lrow) * kbs * 64;
        const uint8_t* sc = stage + static_cast<size_t>(ur) * kbs * 192 + static_cast<size_t>(lrow) * kbs * 16;
        const uint16_t* dd =
            reinterpret_cast<const uint16_t*>(stage + static_cast<size_t>(ur) * kbs * 208) + static_cast<size_t>(lrow) * nb;
        for (; c < c_hi; c += G) {
            const int b = c >> 2, lb = b - b0;
            chunk_q6k(ql + lb * 128, qh + lb * 64, sc + lb * 16, dd + b, b, c & 3, dig, aux, k, acc);
        }
    }
    return acc;
}

// Bytes of one stage per matrix for `rows` rows (Q6_K copies whole 8-row groups).
__host__ __device__ inline size_t rows_bytes(int qt, int rows, int nb) {
    return static_cast<size_t>(rows) * nb * (qt == QT_Q4K ? 144 : 210);
}

// -------------------------------------------------------------- the kernel
// Pro: prepare(float* sm, int k, int tid) fills its scratch (consumers only),
//      value(const float* sm, int i) gives x_i.
// Epi: pre(r0, r1, tid) before the dependency wait (loads of data no kernel
//      of the current step writes), start() after it; with kDeferred, the row results of
//      the CTA go to shared memory and apply(r0, r1, ys, ys2, tid) runs once
//      over all of them with every consumer thread (one memory round trip for
//      the whole CTA); otherwise row(r, v) / row2(r, v0, v1) is called by the
//      lane leading each row group.  finish(float* red, int tid) once per CTA.
template <int QT, bool DUAL, class Pro, class Epi>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemvShape sh, const Pro pro_in, const Epi epi_in) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    uint8_t* dig = smem + off_dig();
    uint8_t* aux = smem + off_aux(sh.k);
    float* psm = reinterpret_cast<float*>(smem + off_pro(QT, sh.k));
    float* ys = reinterpret_cast<float*>(smem + off_ys(QT, sh.k, sh.pro_floats));
    uint8_t* ring = smem + off_ring(QT, sh.k, sh.pro_floats, (DUAL ? 2 : 1) * sh.rows_cta);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();

    // this CTA's rows [r0, r1), in whole 8-row units
    const int u0 = static_cast<int>((static_cast<long long>(blockIdx.x) * sh.units) / gridDim.x);
    const int u1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * sh.units) / gridDim.x);
    const int r0 = 8 * u0, r1 = min(8 * u1, sh.n);
    const int nst = r1 > r0 ? (r1 - r0 + sh.rs - 1) / sh.rs : 0;
    const int S = sh.stages;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // --------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const int nb = sh.nb;
            int issued = 0;
            bool ok = true;
            for (int t = 0; t < nst; ++t) {
                const int slot = t % S;
                if (t >= S && !mbar_wait(&empty[slot], ((t / S) - 1) & 1)) {
                    atomicOr(sh.err, DEVERR_EMPTY_WAIT);
                    ok = false;
                    break;
                }
                const int row0 = r0 + t * sh.rs;
                const int rows = min(sh.rs, r1 - row0);
                uint8_t* st = ring + static_cast<size_t>(slot) * sh.stage_bytes;
                if constexpr (QT == QT_Q4K) {
                    const unsigned bytes = static_cast<unsigned>(rows_bytes(QT, rows, nb));
                    mbar_arrive_expect_tx(&full[slot], DUAL ? 2 * bytes : bytes);
                    bulk_g2s(st, sh.w0 + rows_bytes(QT, row0, nb), bytes, &full[slot], pol);
                    if constexpr (DUAL)
                        bulk_g2s(st + rows_bytes(QT, sh.rs, nb), sh.w1 + rows_bytes(QT, row0, nb), bytes, &full[slot],
                                 pol);
                } else {
                    const int rows8 = (rows + 7) & ~7;
                    const size_t plane = static_cast<size_t>(sh.n8) * nb;
                    const unsigned tot = static_cast<unsigned>(rows_bytes(QT, rows8, nb));
                    mbar_arrive_expect_tx(&full[slot], DUAL ? 2 * tot : tot);
                    const uint8_t* ws[2] = {sh.w0, sh.w1};
#pragma unroll
                    for (int m = 0; m < (DUAL ? 2 : 1); ++m) {
                        const uint8_t* w = ws[m];
                        uint8_t* d = st + m * rows_bytes(QT, sh.rs, nb);
                        const size_t rb = static_cast<size_t>(row0) * nb;
                        bulk_g2s(d, w + rb * 128, rows8 * nb * 128, &full[slot], pol);
                        bulk_g2s(d + static_cast<size_t>(sh.rs) * nb * 128, w + plane * 128 + rb * 64, rows8 * nb * 64,
                                 &full[slot], pol);
                        bulk_g2s(d + static_cast<size_t>(sh.rs) * nb * 192, w + plane * 192 + rb * 16, rows8 * nb * 16,
                                 &full[slot], pol);
                        bulk_g2s(d + static_cast<size_t>(sh.rs) * nb * 208, w + plane * 208 + rb * 2, rows8 * nb * 2,
                                 &full[slot], pol);
                    }
                }
                issued = t + 1;
                if (t == 0) sh.next.issue();  // after this CTA's first stage is on its way
            }
            if (nst == 0) sh.next.issue();
            if (!ok) {
                // do not leave while copies into this CTA's shared memory are in flight
                for (int t = max(0, issued - S); t < issued; ++t)
                    if (!mbar_wait(&full[t % S], (t / S) & 1)) atomicOr(sh.err, DEVERR_DRAIN_WAIT);
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    Pro pro = pro_in;
    Epi epi = epi_in;
    epi.pre(r0, r1, tid);  // inputs of the epilogue that no earlier kernel of this step writes
    pdl_wait();
    pro.prepare(psm, sh.k, tid);
    bar_sync(1, kConsumers);
    build_xrep<QT>(pro, psm, dig, aux, sh.k, warp, lane);
    epi.start();
    bar_sync(1, kConsumers);

    const int G = 1 << sh.lg, rw = 32 / G;
    const int grp = lane >> sh.lg, lg0 = lane & (G - 1);
    const size_t second = rows_bytes(QT, sh.rs, sh.nb);
    for (int t = 0; t < nst; ++t) {
        const int slot = t % S;
        if (!mbar_wait(&full[slot], (t / S) & 1)) {
            atomicOr(sh.err, DEVERR_FULL_WAIT);
            break;
        }
        const uint8_t* st = ring + static_cast<size_t>(slot) * sh.stage_bytes;
        const int row0 = r0 + t * sh.rs;
        const int rows = min(sh.rs, r1 - row0);
        for (int base = warp * rw; base < rows; base += kConsumerWarps * rw) {
            const int lr = base + grp;
            const bool valid = lr < rows;
            float v0 = valid ? row_partial<QT>(st, sh.rs, lr, sh.nb, sh.cr, G, lg0, dig, aux, sh.k) : 0.0f;
            float v1 = 0.0f;
            if constexpr (DUAL)
                v1 = valid ? row_partial<QT>(st + second, sh.rs, lr, sh.nb, sh.cr, G, lg0, dig, aux, sh.k) : 0.0f;
            for (int o = G >> 1; o > 0; o >>= 1) {
                v0 += __shfl_xor_sync(FULL, v0, o);
                if constexpr (DUAL) v1 += __shfl_xor_sync(FULL, v1, o);
            }
            if (valid && lg0 == 0) {
                if constexpr (Epi::kDeferred) {
                    ys[row0 + lr - r0] = v0;
                    if constexpr (DUAL) ys[sh.rows_cta + row0 + lr - r0] = v1;
                } else {
                    if constexpr (DUAL) epi.row2(row0 + lr, v0, v1);
                    else epi.row(row0 + lr, v0);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if constexpr (Epi::kDeferred) {
        bar_sync(1, kConsumers);
        epi.apply(r0, r1, ys, ys + sh.rows_cta, tid);
    }
    epi.finish(psm, tid);
}

// ------------------------------------------------------------- prologues
struct ProPlain {
    const float* x;
    __host__ __device__ int floats(int k) const { return k; }
    __device__ void prepare(float* sm, int k, int tid) {
#pragma unroll 4
        for (int i = 4 * tid; i < k; i += 4 * kConsumers)
            *reinterpret_cast<float4*>(sm + i) = ldcg4(x + i);
    }
    __device__ float value(const float* sm, int i) const { return sm[i]; }
};

// x = RMSNorm(h + y) * w (residual_add_into then rmsnorm_into): the residual
// add of the previous GEMV is done here, by every CTA on its own copy, and
// CTA 0 stores h + y to h_out (the residual stream, double-buffered so that
// no CTA of this kernel reads what CTA 0 writes).  y may be null.  With
// `tok` set, h is row *tok of the embedding table (the step's first layer).
struct ProRmsNorm {
    const float* h;
    const float* y;
    const float* w;
    const int* tok;
    float* h_out;
    float eps;
    int kdim;  // = k
    float r;
    __host__ __device__ int floats(int k) const { return 2 * k + 32; }
    __device__ void prepare(float* sm, int k, int tid) {
        const float* src = h;
        if (tok) src = h + static_cast<size_t>(__ldcg(tok)) * k;
        float ss = 0.0f;
#pragma unroll 4
        for (int i = 4 * tid; i < k; i += 4 * kConsumers) {
            float4 v = ldcg4(src + i);
            if (y) {
                const float4 a = ldcg4(y + i);
                v.x += a.x;
                v.y += a.y;
                v.z += a.z;
                v.w += a.w;
            }
            const float4 ww = __ldg(reinterpret_cast<const float4*>(w + i));
            *reinterpret_cast<float4*>(sm + i) = v;
            *reinterpret_cast<float4*>(sm + k + i) = ww;
            if (h_out && blockIdx.x == 0) *reinterpret_cast<float4*>(h_out + i) = v;
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
        }
        ss = warp_sum(ss);
        float* red = sm + 2 * k;
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        bar_sync(1, kConsumers);
        float tot = 0.0f;
#pragma unroll
        for (int i = 0; i < kConsumerWarps; ++i) tot += red[i];
        r = 1.0f / sqrtf(tot / static_cast<float>(k) + eps);
    }
    __device__ float value(const float* sm, int i) const { return (sm[i] * r) * sm[kdim + i]; }
};

// ------------------------------------------------------------- epilogues
struct EpiBase {
    static constexpr bool kDeferred = true;
    __device__ void pre(int, int, int) {}
    __device__ void start() {}
    __device__ void row(int, float) {}
    __device__ void row2(int, float, float) {}
    __device__ void finish(float*, int) {}
};
struct EpiStore : EpiBase {
    float* y;
    __device__ void apply(int r0, int r1, const float* ys, const float*, int tid) {
        for (int r = r0 + tid; r < r1; r += kConsumers) y[r] = ys[r - r0];
    }
};
struct EpiSwiGlu : EpiBase {  // act = silu(W_gate x) * (W_up x) (fused_swiglu_into)
    float* act;
    __device__ void apply(int r0, int r1, const float* ys, const float* ys2, int tid) {
        for (int r = r0 + tid; r < r1; r += kConsumers) act[r] = silu(ys[r - r0]) * ys2[r - r0];
    }
};

}  // namespace qg
