// GEMV engine for GGUF k-quant weights on GB300 (sm_103a).
//
// y[n] = sum_k deq(W[n][k]) * x[k], one launch per projection (or per pair of
// projections sharing an input), in the role of the float ("mwv") Q4_K /
// Q6_K GEMV of forward_qwen35_cuda.rs (gemv_dispatch, pin_float_gemv).
//
// Arithmetic.  x (K floats, after the kernel's prologue: RMSNorm, gated norm,
// ...) becomes a 24-bit block-fixed-point integer per element: in every
// 256-element block (one k-quant super-block of the weights), n_i =
// rint(x_i * 2^(22-e)) with 2^e <= max|x| < 2^(e+1), so |n_i| < 2^23 and the
// representation keeps the 24 significant bits of the block's largest element
// (f32 keeps 24).  n_i is stored as three byte planes (n = n2*65536 + n1*256 +
// n0, n2 signed); every sum of quant*n over a sub-block is computed EXACTLY
// with dp4a, the sub-block sums of a 64-weight chunk are weighted by their
// integer scales in integer arithmetic, and one float per chunk and row comes
// out.  This is not the int8 activation quantisation forward_qwen35_cuda.rs
// rejects (pin_float_gemv): the only rounding of x is below 2^-23 of its
// block's largest magnitude, and the integer sums carry no rounding at all.
//
//   Q4_K sub-block j (32 weights): d*sc_j*sum(q*x) - dmin*m_j*sum(x)
//   Q6_K group of 16 weights:      d*sc*sum((q-32)*x)
//
// Work split.  K is cut into slices of 32 chunks (64 weights each), then the
// binary digits of the rest (16, 8, 4 chunks).  In a slice of G chunks, G
// lanes cover one row, one chunk each, and every lane keeps the x digits of
// ITS chunk in registers for all the rows it visits, so the inner loop reads
// only weights from shared memory.  A row's value is the sum over slices (in
// slice order) of the G lanes' chunk values reduced by a fixed xor tree.
//
// Memory side.  Each CTA owns a range of whole 8-row groups.  A producer warp
// streams stages of 64 super-block rows (U = 8 * 32/G rows x G/4 blocks of
// the current slice) global -> shared with 1-D bulk copies (cp.async.bulk,
// the TMA engine) into a ring guarded by mbarriers, L2 evict-first.  In the
// grouped layouts (the model's weights) a stage is one contiguous piece per
// 8-row group; raw GGUF Q4_K rows (the building-block entry point) take one
// copy per row when a row spans several slices.  Copies are issued at kernel
// start, before the programmatic-dependent-launch wait, so a kernel's weights
// stream in while the previous kernel finishes.
#pragma once
#include "qg_common.cuh"

namespace qg {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxStages = 8;
constexpr int kMaxSlices = 12;             // K <= 16384
constexpr int QT_Q4K = 12;
constexpr int QT_Q6K = 14;
// Weight layouts.  RAW: GGUF Q4_K rows.  GROUPED: rows padded to a multiple
// of 8; for every 8-row group g and super-block b one group-block of GB
// bytes: Q4_K: the 8 rows' 144-byte blocks (GB = 1152); Q6_K (GB = 1680):
// for row rr and 64-weight quarter cq = 2 half + part (u = 4 rr + cq) a
// 48-byte record at 48u [ql[64 half + 16 part ..16] | ql[64 half + 32 + 16
// part ..16] | qh[16 cq ..16]], the quarter's four scales sc[8 half + part +
// 2s] (s = 0..3) at 1536 + 4u, and the row's fp16 d at 1664 + 2 rr: every
// lane's bytes of a row sit at three fixed offsets.  Group-blocks are stored
// slice-major: the K slices (8 super-blocks each, then 4, 2, 1 for the rest)
// one after the other, inside a slice group by group, so that any run of
// consecutive groups of one slice is one contiguous piece.
constexpr int LAYOUT_RAW = 0;
constexpr int LAYOUT_GROUPED = 1;
constexpr int kStageBlockRows = 64;        // super-block rows per stage
constexpr long long kAbortPollCycles = 100000;  // ~50 us between reads of the abort word in a long wait

__host__ __device__ constexpr int block_bytes(int qt) { return qt == QT_Q4K ? 144 : 210; }
__host__ __device__ constexpr int group_block_bytes(int qt) { return 8 * block_bytes(qt); }
__host__ __device__ constexpr int stage_bytes_of(int qt) { return kStageBlockRows * block_bytes(qt); }

// The K slice holding super-block b: its first block b0 and its width kb.
__host__ __device__ inline void block_slice(int nb, int b, int& b0, int& kb) {
    const int full = nb / 8;
    if (b < 8 * full) {
        b0 = b & ~7;
        kb = 8;
        return;
    }
    int c = 8 * full;
    for (int w = 4; w >= 1; w >>= 1)
        if ((nb - 8 * full) & w) {
            if (b < c + w) {
                b0 = c;
                kb = w;
                return;
            }
            c += w;
        }
    b0 = c;
    kb = 1;
}
// Byte offset of group-block (g, b) in the grouped layout of n8 rows.
__host__ __device__ inline size_t grouped_offset(int n8, int nb, int g, int b, int GB) {
    int b0, kb;
    block_slice(nb, b, b0, kb);
    return (static_cast<size_t>(n8 / 8) * b0 + static_cast<size_t>(g) * kb + (b - b0)) * GB;
}

// Geometry of one launch (identical on host and device).
struct GemvShape {
    const uint8_t* w0;  // first matrix
    const uint8_t* w1;  // second matrix of a dual launch (same shape), else null
    int n, n8, k, nb, cr;
    int nsl;                   // slices
    int sl_c0[kMaxSlices];     // first chunk of each slice
    int sl_lg[kMaxSlices];     // log2(chunks) of each slice (lanes per row)
    int units;                 // ceil(n / 8)
    int pp;                    // row passes per stage (a stage: pp * 64 super-block rows)
    int stages;                // ring depth
    int pro_floats;            // prologue scratch floats
    int rows_cta;              // most rows one CTA owns (row-result buffer)
    float* part;               // split-K mode: slice sums [nsl][n8] (global scratch)
    unsigned* err;
    L2Prefetch next;           // operands of the next kernel, pulled into L2 by the producer
};

// Shared-memory layout offsets.  aux: per 256-element super-block the unit
// 2^(e-22) (float), then Q4_K: per 32-element sub-block the sum of n (float);
// Q6_K: per 16-element group -32 * (sum of n) (float), ordered [block][cq][s].
__host__ __device__ inline int xaux_bytes(int qt, int k) {
    return ((4 * (k / 256) + 15) & ~15) + (qt == QT_Q4K ? 4 * (k / 32) : 4 * (k / 16));
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
// Blocks [b_lo, b_hi) only (default: all), for a CTA that uses just some slices.
template <int QT, class Pro>
__device__ void build_xrep(const Pro& pro, const float* sm, uint8_t* dig, uint8_t* aux, int k, int warp,
                           int lane, int b_lo = 0, int b_hi = -1) {
    const int nsb = b_hi < 0 ? (k >> 8) : b_hi;
    float* units = reinterpret_cast<float*>(aux);
    // a warp's blocks in batches of Pro::kBatch whose global loads are all
    // issued first (load8), so a prologue that reads x from global memory pays
    // one round trip per batch; value8 then turns them into x (every lane of
    // the warp calls it: it may reduce across lanes)
    constexpr int NB = Pro::kBatch;
    for (int bb = b_lo + warp; bb < nsb; bb += NB * kConsumerWarps) {
        typename Pro::Raw raw[NB];
#pragma unroll
        for (int t = 0; t < NB; ++t) {
            const int b = bb + t * kConsumerWarps;
            if (b < nsb) pro.load8(256 * b + 8 * lane, raw[t]);
        }
#pragma unroll
        for (int t = 0; t < NB; ++t) {
            const int b = bb + t * kConsumerWarps;
            if (b >= nsb) break;
            const int i0 = 256 * b + 8 * lane;
            float x[8];
            pro.value8(sm, i0, raw[t], x);
            unsigned am = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) am = max(am, __float_as_uint(x[j]) & 0x7fffffffu);
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
                // the 16-element group of lanes (2i, 2i+1) is group s = (lane & 15) >> 2
                // of quarter cq = 2 half + part of block b: nf at [b][cq][s]
                nsum += __shfl_xor_sync(FULL, nsum, 1);
                if ((lane & 1) == 0) {
                    const int cq = 2 * (lane >> 4) + ((lane >> 1) & 1), sg = (lane & 15) >> 2;
                    reinterpret_cast<float*>(aux + aux_tail(k))[16 * b + 4 * cq + sg] = -32.0f * static_cast<float>(nsum);
                }
            }
        }
    }
}

// ------------------------------------------------------------ chunk digits
// Lane j (0..G-1) of a row in a slice of G chunks covers block bl of the
// slice and quarter q (Q4_K: 64-weight group g; Q6_K: cq = 2 half + part).
// Q6_K lanes are ordered block-fastest so that the 8 lanes of a shared-memory
// phase read different group-blocks.
template <int QT>
__device__ __forceinline__ void lane_chunk(int j, int lg, int& bl, int& q) {
    if constexpr (QT == QT_Q4K) {
        bl = j >> 2;
        q = j & 3;
    } else {
        bl = j & ((1 << (lg - 2)) - 1);
        q = j >> (lg - 2);
    }
}

__device__ __forceinline__ unsigned u4w(const uint4& v, int w) { return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w; }

// x digits of one Q4_K chunk (x[64c, 64c + 64)): planes of the low-nibble
// sub-block (x[64c + 16h ..]) and of the high-nibble one (x[64c + 32 + 16h ..]).
// The dot takes the high nibbles in place (16 x their value: one mask instead
// of a shift and a mask), so every integer sum it forms is 16 x the plain one;
// the sums of n and the unit are kept pre-scaled to match (x16, /16: powers of
// two, so the row value is bit for bit the one of the plain form).
struct DigQ4 {
    uint4 lo[2][3], hi[2][3];
    float ns0, ns1;  // 16 x the sums of n over the two sub-blocks
    float unit;      // 2^(e-22) / 16 of the super-block
};
__device__ __forceinline__ void load_dig_q4(DigQ4& D, int c, const uint8_t* dig, const uint8_t* aux, int k) {
    const int xo = 64 * c;
    const unsigned u0 = static_cast<unsigned>(xo) >> 4;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const unsigned ul = swz(QT_Q4K, u0 + h) << 4, uh = swz(QT_Q4K, u0 + 2 + h) << 4;
#pragma unroll
        for (int p = 0; p < 3; ++p) {
            D.lo[h][p] = *reinterpret_cast<const uint4*>(dig + p * k + ul);
            D.hi[h][p] = *reinterpret_cast<const uint4*>(dig + p * k + uh);
        }
    }
    const float2 ns = *reinterpret_cast<const float2*>(aux + aux_tail(k) + 4 * (xo >> 5));
    D.ns0 = 16.0f * ns.x;
    D.ns1 = 16.0f * ns.y;
    D.unit = 0.0625f * reinterpret_cast<const float*>(aux)[xo >> 8];
}

// One row's Q4_K chunk g of the 144-byte block at blk against the lane's digits.
__device__ __forceinline__ float dot_q4k(const uint8_t* blk, int g, const DigQ4& D) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 16 + 32 * g);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 32 + 32 * g);
    unsigned a0 = 0, a1 = 0, b0 = 0, b1 = 0;
    int a2 = 0, b2 = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint4 q = h ? qb : qa;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const unsigned qw = u4w(q, w);
            const unsigned lo = qw & 0x0f0f0f0fu, hi = qw & 0xf0f0f0f0u;  // hi: 16 x the high nibbles
            a0 = dp4a_uu(lo, u4w(D.lo[h][0], w), a0);
            a1 = dp4a_uu(lo, u4w(D.lo[h][1], w), a1);
            a2 = dp4a_us(lo, u4w(D.lo[h][2], w), a2);
            b0 = dp4a_uu(hi, u4w(D.hi[h][0], w), b0);
            b1 = dp4a_uu(hi, u4w(D.hi[h][1], w), b1);
            b2 = dp4a_us(hi, u4w(D.hi[h][2], w), b2);
        }
    }
    // scale / min of sub-blocks j = 2g (low nibbles) and 2g+1 (high nibbles)
    const float d = f16_to_f32(static_cast<uint16_t>(hdr.x & 0xffffu));
    const float dmin = f16_to_f32(static_cast<uint16_t>(hdr.x >> 16));
    // the 6-bit scale/min of sub-blocks j = 2g, 2g + 1 as shifts and masks:
    // j < 4 (g < 2) is byte j of the scale and min words; j >= 4 is the low /
    // high nibble of byte j + 4 plus the top two bits of byte j - 4
    int sc[2], mn[2];
    const bool low = g < 2;
    const unsigned asc = low ? hdr.y : hdr.w, amn = low ? hdr.z : hdr.w;
    const unsigned msk = low ? 63u : 15u, mhi = low ? 0u : 0x30u, sm4 = low ? 0u : 4u;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const unsigned sh = 16u * static_cast<unsigned>(g & 1) + 8u * t;
        sc[t] = static_cast<int>(((asc >> sh) & msk) | ((hdr.y >> (sh + 2u)) & mhi));
        mn[t] = static_cast<int>(((amn >> (sh + sm4)) & msk) | ((hdr.z >> (sh + 2u)) & mhi));
    }
    // the low sub-block's scale x16 matches the in-place high nibbles: I = 16 x
    // the plain weighted sum, |I| < 2 * 16 * 63 * 15 * 255 * 32 < 2^31, and each
    // I is 16 x an integer below 2^24 in magnitude, so it converts to f32 exactly
    const int s0 = sc[0] << 4;
    const int I0 = s0 * static_cast<int>(a0) + sc[1] * static_cast<int>(b0);
    const int I1 = s0 * static_cast<int>(a1) + sc[1] * static_cast<int>(b1);
    const int I2 = s0 * a2 + sc[1] * b2;
    const float F = fmaf(static_cast<float>(I2), 65536.0f, fmaf(static_cast<float>(I1), 256.0f, static_cast<float>(I0)));
    const float M = fmaf(static_cast<float>(mn[0]), D.ns0, static_cast<float>(mn[1]) * D.ns1);
    return D.unit * fmaf(d, F, -(dmin * M));
}

// x digits of one Q6_K quarter (block b, cq = 2 half + part): the four
// 16-element groups x[256b + 128 half + 32 s + 16 part ..], s = 0..3, and
// nf[s] = -32 * (sum of n over group s) as a float (the -32 offset of the
// quants, applied once per group instead of per weight).
struct DigQ6 {
    uint4 d[4][3];
    float nf[4];
    float unit;
};
__device__ __forceinline__ void load_dig_q6(DigQ6& D, int b, int cq, const uint8_t* dig, const uint8_t* aux, int k) {
    const int half = cq >> 1, part = cq & 1;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int pos = 256 * b + 128 * half + 32 * s + 16 * part;
        const unsigned u = swz(QT_Q6K, static_cast<unsigned>(pos) >> 4);
#pragma unroll
        for (int p = 0; p < 3; ++p) D.d[s][p] = *reinterpret_cast<const uint4*>(dig + p * k + (u << 4));
    }
    const float4 nf = reinterpret_cast<const float4*>(aux + aux_tail(k))[4 * b + cq];
    D.nf[0] = nf.x;
    D.nf[1] = nf.y;
    D.nf[2] = nf.z;
    D.nf[3] = nf.w;
    D.unit = reinterpret_cast<const float*>(aux)[b];
}

// One row's Q6_K quarter.  rec: its 48-byte record [A | B | H] (A = ql[64
// half + 16 part ..], B = ql[64 half + 32 + 16 part ..], H = qh[16 cq ..]);
// S: its four int8 scales (group s in byte s); dbits: its fp16 d.
// value = d * unit * sum_s sc_s * (sum_i q_i n_i - 32 * sum_i n_i), the first
// sum exact in integers per digit plane, the second from nf.
__device__ __forceinline__ float dot_q6k(const uint8_t* rec, unsigned S, uint16_t dbits, const DigQ6& D) {
    const uint4 A = *reinterpret_cast<const uint4*>(rec);
    const uint4 B = *reinterpret_cast<const uint4*>(rec + 16);
    const uint4 H = *reinterpret_cast<const uint4*>(rec + 32);
    int I0 = 0, I1 = 0, I2 = 0;
    float C = 0.0f;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        unsigned t0 = 0u, t1 = 0u;
        int t2 = 0;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const unsigned a = u4w(A, w), bb = u4w(B, w), hh = u4w(H, w);
            unsigned q;
            if (s == 0) q = (a & 0x0f0f0f0fu) | ((hh << 4) & 0x30303030u);
            else if (s == 1) q = (bb & 0x0f0f0f0fu) | ((hh << 2) & 0x30303030u);
            else if (s == 2) q = ((a >> 4) & 0x0f0f0f0fu) | (hh & 0x30303030u);
            else q = ((bb >> 4) & 0x0f0f0f0fu) | ((hh >> 2) & 0x30303030u);
            t0 = dp4a_uu(q, u4w(D.d[s][0], w), t0);
            t1 = dp4a_uu(q, u4w(D.d[s][1], w), t1);
            t2 = dp4a_us(q, u4w(D.d[s][2], w), t2);
        }
        const int sc = static_cast<int>(S << (24 - 8 * s)) >> 24;  // byte s, sign-extended
        // |sc * t| <= 128 * 63 * 255 * 16 per group, four groups: fits in int32
        I0 += sc * static_cast<int>(t0);
        I1 += sc * static_cast<int>(t1);
        I2 += sc * t2;
        C = fmaf(static_cast<float>(sc), D.nf[s], C);
    }
    const float F = fmaf(static_cast<float>(I2), 65536.0f, fmaf(static_cast<float>(I1), 256.0f, static_cast<float>(I0))) + C;
    return (f16_to_f32(dbits) * D.unit) * F;
}

// ----------------------------------------------------------------- pipe
// A ring of stages in shared memory between the producer warp and the
// consumer warps: `full` completes when a stage's bulk copies have landed,
// `empty` when all consumer warps released it.  q counts the stages taken
// (the same sequence on both sides).  Waits are bounded and also give up
// once `abort` (the kernel's error word) is non-zero, so a failed pipeline
// ends in about one wait.
struct Pipe {
    uint64_t* full;
    uint64_t* empty;
    uint8_t* base;
    int ns;
    int slot_bytes;
    unsigned q;        // stages taken so far
    unsigned* err;
    unsigned* abort;
    int lane;
    uint64_t pol;
    int slot = 0;      // q % ns, kept incrementally (no division on the hot path)
    unsigned ph = 0;   // (q / ns) & 1
    __device__ uint8_t* cur() const { return base + static_cast<size_t>(slot) * slot_bytes; }
    __device__ void advance() {
        ++q;
        if (++slot == ns) {
            slot = 0;
            ph ^= 1u;
        }
    }
    // The abort word is read only once a wait has lasted ~50 us (then every
    // ~50 us): a load of it on every missed poll would put an L2 round trip on
    // the critical path of each stage that lands just in time.
    __device__ bool wait_bar(uint64_t* bar, unsigned parity) const {
        if (mbar_try_wait(bar, parity)) return true;
        const long long t0 = clock64();
        long long check = t0 + kAbortPollCycles;
        while (!mbar_try_wait(bar, parity)) {
            const long long now = clock64();
            if (now - t0 > kWaitCycles) return false;
            if (now > check) {
                if (__ldcg(abort)) return false;
                check = now + kAbortPollCycles;
            }
        }
        return true;
    }
    __device__ void fail(unsigned bit) const {
        atomicOr(err, bit);
    }
    // consumer side (every lane of every consumer warp)
    __device__ void wait_full() const {
        if (!wait_bar(&full[slot], ph) && lane == 0) fail(DEVERR_FULL_WAIT);
    }
    __device__ void release() {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        advance();
    }
    // producer side (the whole producer warp)
    __device__ bool acquire() {
        int good = 1;
        if (lane == 0 && q >= static_cast<unsigned>(ns)) good = wait_bar(&empty[slot], ph ^ 1u) ? 1 : 0;
        good = __shfl_sync(FULL, good, 0);
        if (!good && lane == 0) fail(DEVERR_EMPTY_WAIT);
        return good != 0;
    }
    __device__ void expect(unsigned bytes) {
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], bytes);
        __syncwarp();
    }
    __device__ void copy(void* dst, const void* src, unsigned bytes) { bulk_g2s(dst, src, bytes, &full[slot], pol); }
    __device__ void commit() { advance(); }
    // error exit: wait (bounded) for this CTA's copies still in flight
    __device__ void drain() {
        if (lane != 0) return;
        const unsigned lo = q > static_cast<unsigned>(ns) ? q - ns : 0u;
        for (unsigned t = lo; t < q; ++t) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&full[t % ns], (t / ns) & 1u))
                if (clock64() - t0 > kWaitCycles) {
                    atomicOr(err, DEVERR_DRAIN_WAIT);
                    break;
                }
        }
    }
};

// Sum of v over the G lanes of its row group (xor tree, G a power of two <= 32).
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        if (o < G) v += __shfl_xor_sync(FULL, v, o);
    return v;
}

// The lane's share of one stage row pass in a slice of G = 2^LG chunks: its
// byte offsets inside the stage (constant for the slice: row rl of the pass,
// block bl of the slice, quarter q), and one pass's bytes (64 block-rows).
template <int QT, int LAYOUT, int LG>
struct LaneRow {
    static constexpr int kb = (1 << LG) >> 2;
    static constexpr int GB = group_block_bytes(QT);
    static constexpr int pass_bytes = kStageBlockRows * block_bytes(QT);
    int o0, o1, o2, o3;  // Q4_K: block; Q6_K: [A | B | H] record, scale record, d
    int q;
    __device__ __forceinline__ LaneRow(int rl, int bl, int q_) : q(q_) {
        if constexpr (QT == QT_Q4K) {
            o0 = LAYOUT == LAYOUT_GROUPED ? ((rl >> 3) * kb + bl) * GB + (rl & 7) * 144 : (rl * kb + bl) * 144;
            o1 = o2 = o3 = 0;
        } else {  // records of the planar Q6_K group-block (see the layout note at the top)
            const int base = ((rl >> 3) * kb + bl) * GB, rr = rl & 7, u = 4 * rr + q;
            o0 = base + 48 * u;
            o1 = base + 1536 + 4 * u;
            o2 = base + 1664 + 2 * rr;
            o3 = 0;
        }
    }
    // the lane's chunk value of its row in the pass starting at ps, summed
    // over the row's G lanes (lanes of rows past the range read stale bytes
    // inside the slot; their sums are not stored)
    __device__ __forceinline__ float value(const uint8_t* ps, const DigQ4& d4, const DigQ6& d6) const {
        float v;
        if constexpr (QT == QT_Q4K) v = dot_q4k(ps + o0, q, d4);
        else v = dot_q6k(ps + o0, *reinterpret_cast<const unsigned*>(ps + o1), *reinterpret_cast<const uint16_t*>(ps + o2), d6);
        return group_sum<(1 << LG)>(v);
    }
};

// The lane's chunk digits for slice s (lanes per row 2^LG).
template <int QT, int LG>
__device__ __forceinline__ void slice_lane(const GemvShape& sh, int s, int lane, const uint8_t* dig, const uint8_t* aux,
                                           int k, int& bl, int& q, DigQ4& d4, DigQ6& d6) {
    lane_chunk<QT>(lane & ((1 << LG) - 1), LG, bl, q);
    const int b = (sh.sl_c0[s] >> 2) + bl;
    if constexpr (QT == QT_Q4K) load_dig_q4(d4, 4 * b + q, dig, aux, k);
    else load_dig_q6(d6, b, q, dig, aux, k);
}

// Rows [r0, r1) of a launch with `units` 8-row units over gridDim.x CTAs.
__device__ __forceinline__ void cta_rows(int units, int n, int& r0, int& r1) {
    const int u0 = static_cast<int>((static_cast<long long>(blockIdx.x) * units) / gridDim.x);
    const int u1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * units) / gridDim.x);
    r0 = 8 * u0;
    r1 = min(8 * u1, n);
}

// ---------------------------------------------------------------- producer
// Stages in consumption order: slices, then passes of U = 8 * 32/G rows,
// then the matrices of a dual launch.  `next` (if any) is issued once this
// CTA's first stage is on its way.
template <int QT, int LAYOUT, bool DUAL>
__device__ bool gemv_produce(Pipe& p, const GemvShape& sh, const uint8_t* w0, const uint8_t* w1, int r0, int r1,
                             const L2Prefetch* next) {
    constexpr int GB = group_block_bytes(QT);
    const int nb = sh.nb;
    bool first = true;
    for (int s = 0; s < sh.nsl; ++s) {
        const int lg = sh.sl_lg[s], kb = (1 << lg) >> 2, U = (256 >> lg) * sh.pp, b0 = sh.sl_c0[s] >> 2;
        for (int row0 = r0; row0 < r1; row0 += U) {
            const int rows = min(U, r1 - row0);
#pragma unroll
            for (int m = 0; m < (DUAL ? 2 : 1); ++m) {
                if (!p.acquire()) return false;
                const uint8_t* w = m ? w1 : w0;
                uint8_t* st = p.cur();
                if constexpr (LAYOUT == LAYOUT_GROUPED) {
                    // consecutive groups of one slice: one contiguous piece
                    const unsigned bytes = static_cast<unsigned>((rows + 7) >> 3) * kb * GB;
                    p.expect(bytes);
                    if (p.lane == 0)
                        p.copy(st, w + (static_cast<size_t>(sh.n8 / 8) * b0 + static_cast<size_t>(row0 >> 3) * kb) * GB,
                               bytes);
                } else {  // raw Q4_K rows
                    if (kb == nb) {
                        const unsigned bytes = static_cast<unsigned>(rows) * nb * 144u;
                        p.expect(bytes);
                        if (p.lane == 0) p.copy(st, w + static_cast<size_t>(row0) * nb * 144, bytes);
                    } else {
                        const unsigned piece = static_cast<unsigned>(kb) * 144u;
                        p.expect(rows * piece);
                        for (int i = p.lane; i < rows; i += 32)
                            p.copy(st + static_cast<size_t>(i) * piece,
                                   w + (static_cast<size_t>(row0 + i) * nb + b0) * 144, piece);
                    }
                }
                p.commit();
                if (first && next && p.lane == 0) next->issue();
                first = false;
            }
        }
    }
    if (first && next && p.lane == 0) next->issue();
    return true;
}

// --------------------------------------------------------------- consumer
// Slice s (2^LG lanes per row) of the rows [r0, r1): every stage of pp passes
// of U rows; lane j == 0 of each row adds the row's slice sum to ys (ys2 for
// the second matrix of a dual launch), in slice order.
template <int QT, int LAYOUT, bool DUAL, int LG>
__device__ void consume_slice(Pipe& p, const GemvShape& sh, int s, int r0, int r1, float* ys, float* ys2,
                              const uint8_t* dig, const uint8_t* aux, int warp, int lane) {
    constexpr int rpw = 32 >> LG, U = 8 * rpw;
    const int rl = warp * rpw + (lane >> LG);
    const bool lead = (lane & ((1 << LG) - 1)) == 0;
    int bl, q;
    DigQ4 d4;
    DigQ6 d6;
    slice_lane<QT, LG>(sh, s, lane, dig, aux, sh.k, bl, q, d4, d6);
    const LaneRow<QT, LAYOUT, LG> lr(rl, bl, q);
    const int pp = sh.pp;
    for (int row0 = r0; row0 < r1; row0 += U * pp) {
        const int npass = min(pp, (r1 - row0 + U - 1) / U);  // passes holding rows of the range
#pragma unroll
        for (int m = 0; m < (DUAL ? 2 : 1); ++m) {
            p.wait_full();
            const uint8_t* ps = p.cur();
            float* y = (m ? ys2 : ys) + (row0 - r0) + rl;
            for (int pass = 0; pass < npass; ++pass, ps += lr.pass_bytes, y += U) {
                const float v = lr.value(ps, d4, d6);
                if (lead && row0 + pass * U + rl < r1) *y = s ? *y + v : v;
            }
            p.release();
        }
    }
}

// Pro: pre(float* sm, int k, int tid) before the dependency wait (inputs no
//      earlier kernel of the step writes; called by the kernel),
//      prepare(float* sm, int k, int tid) fills the rest of its scratch,
//      load8(i0, Raw&) issues the global loads behind x_i0 .. x_i0+7 (i0 % 8
//      == 0) and value8(sm, i0, const Raw&, float* v) gives those 8 values;
//      kBatch: blocks whose loads build_xrep keeps in flight per warp.
// Epi: pre(r0, r1, tid) before the dependency wait (loads of data no kernel of
//      the current step writes; called by the kernel), start() after the
//      prologue, apply(r0, r1, ys, ys2, tid) once over the CTA's row results
//      with every consumer thread, finish(float* red, int tid) once per CTA.
template <int QT, int LAYOUT, bool DUAL, class Pro, class Epi>
__device__ void gemv_consume(Pipe& p, const GemvShape& sh, int r0, int r1, Pro& pro, Epi& epi, uint8_t* smem,
                             int tid) {
    const int warp = tid >> 5, lane = tid & 31, k = sh.k;
    uint8_t* dig = smem + off_dig();
    uint8_t* aux = smem + off_aux(k);
    float* psm = reinterpret_cast<float*>(smem + off_pro(QT, k));
    float* ys = reinterpret_cast<float*>(smem + off_ys(QT, k, sh.pro_floats));
    float* ys2 = ys + sh.rows_cta;
    pro.prepare(psm, k, tid);
    bar_sync(1, kConsumers);
    build_xrep<QT>(pro, psm, dig, aux, k, warp, lane);
    epi.start();
    bar_sync(1, kConsumers);

    for (int s = 0; s < sh.nsl; ++s) {
        switch (sh.sl_lg[s]) {
            case 5: consume_slice<QT, LAYOUT, DUAL, 5>(p, sh, s, r0, r1, ys, ys2, dig, aux, warp, lane); break;
            case 4: consume_slice<QT, LAYOUT, DUAL, 4>(p, sh, s, r0, r1, ys, ys2, dig, aux, warp, lane); break;
            case 3: consume_slice<QT, LAYOUT, DUAL, 3>(p, sh, s, r0, r1, ys, ys2, dig, aux, warp, lane); break;
            default: consume_slice<QT, LAYOUT, DUAL, 2>(p, sh, s, r0, r1, ys, ys2, dig, aux, warp, lane); break;
        }
        bar_sync(1, kConsumers);  // this slice's row sums are in before the next adds to them
    }
    epi.apply(r0, r1, ys, ys2, tid);
    epi.finish(psm, tid);
}

// ------------------------------------------------------------- the kernel
// The two engine kernels (and their launchers) have internal linkage: every
// translation unit registers its own device copy of a kernel it instantiates,
// so an instantiation shared by two units must not be merged into one host
// stub whose shared-memory attribute was set on the other unit's copy.
namespace {

template <int QT, int LAYOUT, bool DUAL, class Pro, class Epi>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemvShape sh, const Pro pro_in, const Epi epi_in) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();
    int r0, r1;
    cta_rows(sh.units, sh.n, r0, r1);
    if (tid == 0) {
        for (int s = 0; s < sh.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    // the kernel's error word doubles as its abort flag
    Pipe p{full, empty, smem + off_ring(QT, sh.k, sh.pro_floats, (DUAL ? 2 : 1) * sh.rows_cta), sh.stages,
           sh.pp * stage_bytes_of(QT), 0u, sh.err, sh.err, lane, 0ull};
    if (warp == kConsumerWarps) {
        p.pol = policy_evict_first();
        if (!gemv_produce<QT, LAYOUT, DUAL>(p, sh, sh.w0, sh.w1, r0, r1, &sh.next)) p.drain();
        return;
    }
    Pro pro = pro_in;
    Epi epi = epi_in;
    epi.pre(r0, r1, tid);  // inputs that no earlier kernel of this step writes
    pro.pre(reinterpret_cast<float*>(smem + off_pro(QT, sh.k)), sh.k, tid);
    pdl_wait();
    gemv_consume<QT, LAYOUT, DUAL>(p, sh, r0, r1, pro, epi, smem, tid);
}

}  // namespace

// ------------------------------------------------------------ split-K mode
// For GEMVs with few rows and several K slices (ffn_down, the output
// projections) one CTA per row group would run its slices one after another.
// Here the work is (slice, 8-row group) tasks, slice-major, spread evenly over
// the CTAs; a CTA's consecutive tasks of one slice stream as contiguous
// stages.  Each task writes its rows' slice sums to part[slice][row]; the
// consumer of y (the next RMSNorm prologue, or the residual add) adds the
// slices in slice order -- the order of the one-CTA-per-row path, so both give
// the same floats -- which saves this kernel an arrival count and a second
// pass over the sums.
// (units * nsl < 2^21 for n <= 2^20 rows and K <= 16384: the products fit in 32 bits)
__device__ __forceinline__ void split_range(const GemvShape& sh, int& t0, int& t1) {
    const unsigned T = static_cast<unsigned>(sh.units) * sh.nsl;
    t0 = static_cast<int>(blockIdx.x * T / gridDim.x);
    t1 = static_cast<int>((blockIdx.x + 1) * T / gridDim.x);
}

template <int QT>
__device__ bool gemv_split_produce(Pipe& p, const GemvShape& sh, const L2Prefetch* next) {
    constexpr int GB = group_block_bytes(QT);
    int t0, t1;
    split_range(sh, t0, t1);
    bool first = true;
    for (int t = t0; t < t1;) {
        const int s = t / sh.units, g = t - s * sh.units;
        const int ge = min(sh.units, g + (t1 - t));
        const int lg = sh.sl_lg[s], kb = (1 << lg) >> 2, U = (256 >> lg) * sh.pp, b0 = sh.sl_c0[s] >> 2;
        const int ra = 8 * g, rb = min(8 * ge, sh.n);
        for (int row0 = ra; row0 < rb; row0 += U) {
            const int rows = min(U, rb - row0);
            if (!p.acquire()) return false;
            const unsigned bytes = static_cast<unsigned>((rows + 7) >> 3) * kb * GB;
            p.expect(bytes);
            if (p.lane == 0)
                p.copy(p.cur(), sh.w0 + (static_cast<size_t>(sh.n8 / 8) * b0 + static_cast<size_t>(row0 >> 3) * kb) * GB,
                       bytes);
            p.commit();
            if (first && next && p.lane == 0) next->issue();
            first = false;
        }
        t += ge - g;
    }
    if (first && next && p.lane == 0) next->issue();
    return true;
}

// Rows [ra, rb) of slice s (2^LG lanes per row): their slice sums to part[s].
template <int QT, int LG>
__device__ void split_slice(Pipe& p, const GemvShape& sh, int s, int ra, int rb, const uint8_t* dig,
                            const uint8_t* aux, int warp, int lane) {
    constexpr int rpw = 32 >> LG, U = 8 * rpw;
    const int rl = warp * rpw + (lane >> LG);
    const bool lead = (lane & ((1 << LG) - 1)) == 0;
    int bl, q;
    DigQ4 d4;
    DigQ6 d6;
    slice_lane<QT, LG>(sh, s, lane, dig, aux, sh.k, bl, q, d4, d6);
    const LaneRow<QT, LAYOUT_GROUPED, LG> lr(rl, bl, q);
    const int pp = sh.pp;
    for (int row0 = ra; row0 < rb; row0 += U * pp) {
        const int npass = min(pp, (rb - row0 + U - 1) / U);
        p.wait_full();
        const uint8_t* ps = p.cur();
        float* y = sh.part + static_cast<size_t>(s) * sh.n8 + row0 + rl;
        for (int pass = 0; pass < npass; ++pass, ps += lr.pass_bytes, y += U) {
            const float v = lr.value(ps, d4, d6);
            if (lead && row0 + pass * U + rl < rb) *y = v;
        }
        p.release();
    }
}

template <int QT, class Pro>
__device__ void gemv_split_consume(Pipe& p, const GemvShape& sh, Pro& pro, uint8_t* smem, int tid) {
    const int warp = tid >> 5, lane = tid & 31, k = sh.k;
    uint8_t* dig = smem + off_dig();
    uint8_t* aux = smem + off_aux(k);
    float* psm = reinterpret_cast<float*>(smem + off_pro(QT, k));
    int t0, t1;
    split_range(sh, t0, t1);
    pro.prepare(psm, k, tid);
    bar_sync(1, kConsumers);
    if (t1 > t0) {  // digits of the slices this CTA's tasks use
        const int s0 = t0 / sh.units, s1 = (t1 - 1) / sh.units;
        build_xrep<QT>(pro, psm, dig, aux, k, warp, lane, sh.sl_c0[s0] >> 2,
                       (sh.sl_c0[s1] + (1 << sh.sl_lg[s1])) >> 2);
    }
    bar_sync(1, kConsumers);
    for (int t = t0; t < t1;) {
        const int s = t / sh.units, g = t - s * sh.units;
        const int ge = min(sh.units, g + (t1 - t));
        const int ra = 8 * g, rb = min(8 * ge, sh.n);
        switch (sh.sl_lg[s]) {
            case 5: split_slice<QT, 5>(p, sh, s, ra, rb, dig, aux, warp, lane); break;
            case 4: split_slice<QT, 4>(p, sh, s, ra, rb, dig, aux, warp, lane); break;
            case 3: split_slice<QT, 3>(p, sh, s, ra, rb, dig, aux, warp, lane); break;
            default: split_slice<QT, 2>(p, sh, s, ra, rb, dig, aux, warp, lane); break;
        }
        t += ge - g;
    }
}

namespace {

template <int QT, class Pro>
__global__ void __launch_bounds__(kThreads, 2) gemv_split_kernel(const GemvShape sh, const Pro pro_in) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < sh.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    Pipe p{full, empty, smem + off_ring(QT, sh.k, sh.pro_floats, 0), sh.stages, sh.pp * stage_bytes_of(QT), 0u,
           sh.err, sh.err, lane, 0ull};
    if (warp == kConsumerWarps) {
        p.pol = policy_evict_first();
        if (!gemv_split_produce<QT>(p, sh, &sh.next)) p.drain();
        return;
    }
    Pro pro = pro_in;
    pro.pre(reinterpret_cast<float*>(smem + off_pro(QT, sh.k)), sh.k, tid);
    pdl_wait();
    gemv_split_consume<QT>(p, sh, pro, smem, tid);
}

}  // namespace

// ------------------------------------------------------------- prologues
// x read straight from global memory by build_xrep (written by an earlier
// kernel or phase: L2 only); no shared-memory copy, so the ring keeps its room.
// Its 16 scratch floats are the epilogue's reduction space (finish).
struct ProPlainG {
    const float* x;
    struct Raw {
        float4 a, b;
    };
    static constexpr int kBatch = 4;
    __host__ __device__ int floats(int) const { return 16; }
    __device__ void pre(float*, int, int) {}
    __device__ void prepare(float*, int, int) {}
    __device__ void load8(int i0, Raw& r) const {
        r.a = ldcg4(x + i0);
        r.b = ldcg4(x + i0 + 4);
    }
    __device__ void value8(const float*, int, const Raw& r, float* v) const {
        v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w;
        v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
    }
};

// x = RMSNorm(h + y) * w (residual_add_into then rmsnorm_into): the residual
// add of the previous GEMV is done here (y given as the previous GEMV's
// slice sums when it ran split-K: summed first, in slice order), by every
// CTA on its own copy, and
// CTA 0 stores h + y to h_out (the residual stream, double-buffered so that
// no CTA of this kernel reads what CTA 0 writes).  y may be null.  With
// `tok` set, h is row *tok of the embedding table (the step's first layer).
struct ProRmsNorm {
    const float* h;
    const float* y;    // y_parts vectors y_stride floats apart, added in order (split-K slice sums)
    const float* w;
    const int* tok;
    float* h_out;
    float eps;
    int kdim;  // = k
    int y_parts, y_stride;
    float r;
    struct Raw {};  // x is staged in shared memory by prepare
    static constexpr int kBatch = 4;
    __host__ __device__ int floats(int k) const { return 2 * k + 32; }
    // the norm weights do not depend on the previous kernel: staged before its wait
    __device__ void pre(float* sm, int k, int tid) {
#pragma unroll 4
        for (int i = 4 * tid; i < k; i += 4 * kConsumers)
            *reinterpret_cast<float4*>(sm + k + i) = __ldg(reinterpret_cast<const float4*>(w + i));
    }
    __device__ void prepare(float* sm, int k, int tid) {
        const float* src = h;
        if (tok) src = h + static_cast<size_t>(__ldcg(tok)) * k;
        float ss = 0.0f;
#pragma unroll 4
        for (int i = 4 * tid; i < k; i += 4 * kConsumers) {
            float4 v = ldcg4(src + i);
            if (y) {
                float4 a = ldcg4(y + i);
                for (int p = 1; p < y_parts; ++p) {
                    const float4 b = ldcg4(y + static_cast<size_t>(p) * y_stride + i);
                    a.x += b.x;
                    a.y += b.y;
                    a.z += b.z;
                    a.w += b.w;
                }
                v.x += a.x;
                v.y += a.y;
                v.z += a.z;
                v.w += a.w;
            }
            *reinterpret_cast<float4*>(sm + i) = v;
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
    __device__ void load8(int, Raw&) const {}
    __device__ void value8(const float* sm, int i0, const Raw&, float* v) const {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float4 a = *reinterpret_cast<const float4*>(sm + i0 + 4 * h);
            const float4 w4 = *reinterpret_cast<const float4*>(sm + kdim + i0 + 4 * h);
            v[4 * h + 0] = (a.x * r) * w4.x;
            v[4 * h + 1] = (a.y * r) * w4.y;
            v[4 * h + 2] = (a.z * r) * w4.z;
            v[4 * h + 3] = (a.w * r) * w4.w;
        }
    }
};

// ------------------------------------------------------------- epilogues
struct EpiBase {
    __device__ void pre(int, int, int) {}
    __device__ void start() {}
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
