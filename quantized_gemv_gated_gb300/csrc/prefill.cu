// Batched prompt prefill: a chunk of prompt tokens goes through every layer
// together, so each projection is one multi-token GEMM on the tensor cores
// (tcgen05.mma) that reads its weights once per chunk instead of once per
// token (the decode session's batched prefill, forward_qwen35_cuda.rs).  The recurrences stay exact token-by-token
// recurrences inside one kernel per layer: the causal conv scans each channel
// over the chunk, the delta rule walks the chunk with each warp's four state
// rows in registers, and the attention of token p reads the cache rows
// 0..pos0+p (causal).  The state it leaves (conv windows, recurrent states, K/V
// rows, the residual stream) is the state the token-by-token decode leaves,
// and the lm_head argmax of the last token is the first generated token.
//
// The same pass runs the batched decode (the decode session's batched decode):
// its columns are split into segments, one per sequence, each with that
// sequence's state and positions, so a lockstep step of n sequences is n
// single-column segments; with at most 8 columns the projections use a
// small-batch GEMV that reads each weight once per group of 4, and a fixed set
// of sequences can replay the whole step as one captured graph (qg_batch_*).
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <type_traits>

#include "qg_layers.cuh"

namespace qg {
namespace {

constexpr int kPfChunk = 1024;  // prompt tokens per pass through the layers
constexpr int kPfMaxSplit = 16; // K splits of a projection (in 64-weight quarters)
constexpr int kAttnSplits = 16; // key splits of a batched decode step's attention
constexpr int kSmallBatch = 8;  // columns of a batched decode step on the small-batch GEMV (groups of 4)

// The columns of one pass split into segments: segment s is one sequence's
// run of consecutive positions pos0[s].. in columns col0[s]..col0[s+1]-1, with
// that sequence's state of the current layer (conv window and recurrent
// state, or K/V cache).  A prefill is one segment; a batched decode step is
// one single-column segment per sequence.
constexpr int kMaxSeg = 16;
struct Segs {
    int n;
    int col0[kMaxSeg + 1];
    const int* pos0;       // device: first position of each segment (so a captured pass replays with new ones)
    int max_seq[kMaxSeg];  // the sequence's cache length (the record stride of a quantized cache)
    float* conv[kMaxSeg];
    float* ssm[kMaxSeg];
    float* kc[kMaxSeg];
    float* vc[kMaxSeg];
};
__device__ __forceinline__ int seg_of(const Segs& sg, int p) {
    int s = 0;
    while (s + 1 < sg.n && p >= sg.col0[s + 1]) ++s;
    return s;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
    return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}
__device__ __forceinline__ int byte_of(const uint4& v, int b) { return (word_of(v, b >> 2) >> (8 * (b & 3))) & 0xff; }

// Raw bytes one thread dequantizes: 16 weights of a 64-weight quarter q of a
// row, part (0..3) = 2 hf + p: weights 64 q + 32 hf + 16 p .. + 15, loaded a
// quarter ahead.  Q4_K: the row's 16-byte block head (d, dmin, the 12 bytes of
// 6-bit scales and mins) and the 16 bytes of nibbles holding those weights
// (low nibbles for hf = 0, high for hf = 1).  Q6_K: the row's 48-byte planar
// record of those weights, its 4 scales and d.
struct RawQ4 {
    uint4 h, q;
};
struct RawQ6 {
    uint4 r[3];
    uint32_t sc;
    uint32_t d;
};

__device__ __forceinline__ void raw_load(const uint8_t* gb, int rr, int q, int part, RawQ4& r) {
    const uint8_t* blk = gb + 144 * rr;
    r.h = *reinterpret_cast<const uint4*>(blk);
    r.q = *reinterpret_cast<const uint4*>(blk + 16 + 32 * q + 16 * (part & 1));
}
__device__ __forceinline__ void raw_load(const uint8_t* gb, int rr, int q, int part, RawQ6& r) {
    const int u = 4 * rr + 2 * (q >> 1) + (part & 1);
#pragma unroll
    for (int w = 0; w < 3; ++w) r.r[w] = *reinterpret_cast<const uint4*>(gb + 48 * u + 16 * w);
    r.sc = *reinterpret_cast<const uint32_t*>(gb + 1536 + 4 * u);
    r.d = *reinterpret_cast<const uint16_t*>(gb + 1664 + 2 * rr);
}

// Q4_K: d * scale_j * nibble - dmin * min_j for sub-block j = 2 q + hf.
__device__ __forceinline__ void raw_decode(const RawQ4& r, int q, int part, float* v) {
    const int hf = part >> 1, j = 2 * q + hf;
    const float d = f16_to_f32(static_cast<uint16_t>(r.h.x & 0xffffu));
    const float dmin = f16_to_f32(static_cast<uint16_t>(r.h.x >> 16));
    int s, m;  // 6-bit scale and min of sub-block j from the 12 bytes at 4..15
    if (j < 4) {
        s = byte_of(r.h, 4 + j) & 63;
        m = byte_of(r.h, 8 + j) & 63;
    } else {
        s = (byte_of(r.h, 8 + j) & 15) | ((byte_of(r.h, j) >> 6) << 4);
        m = (byte_of(r.h, 8 + j) >> 4) | ((byte_of(r.h, 4 + j) >> 6) << 4);
    }
    const float ds = d * static_cast<float>(s), dm = dmin * static_cast<float>(m);
    const int sh = 4 * hf;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int nib = (word_of(r.q, i >> 2) >> (8 * (i & 3) + sh)) & 15;
        v[i] = ds * static_cast<float>(nib) - dm;
    }
}

// Q6_K (planar): weights 128 h + 32 s + 16 p + i (h = q / 2, s = 2 (q & 1) +
// hf, i < 16) are byte i of record (rr, 2 h + p) with its scale s:
// d * scale * (6-bit code - 32).
__device__ __forceinline__ void raw_decode(const RawQ6& r, int q, int part, float* v) {
    const int s = 2 * (q & 1) + (part >> 1);
    const float d = f16_to_f32(static_cast<uint16_t>(r.d & 0xffffu));
    const float ds = d * static_cast<float>(static_cast<int8_t>((r.sc >> (8 * s)) & 0xffu));
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int a = (word_of(r.r[0], i >> 2) >> (8 * (i & 3))) & 0xff;
        const int b = (word_of(r.r[1], i >> 2) >> (8 * (i & 3))) & 0xff;
        const int hb = (word_of(r.r[2], i >> 2) >> (8 * (i & 3))) & 0xff;
        int code;
        if (s == 0) code = (a & 15) | ((hb & 3) << 4);
        else if (s == 1) code = (b & 15) | (((hb >> 2) & 3) << 4);
        else if (s == 2) code = (a >> 4) | (((hb >> 4) & 3) << 4);
        else code = (b >> 4) | (((hb >> 6) & 3) << 4);
        v[i] = ds * static_cast<float>(code - 32);
    }
}

// ------------------------------------------- prefill GEMM on the tensor cores
// Y = W X for a chunk of P > 8 tokens with tcgen05.mma: the CTA's 128 weight
// rows are the A operand (M = 128), its 256 tokens (two 128-token tiles) the B
// operand (N = 256, or 128 where the second tile holds no token), both K-major
// bf16 tiles in shared memory, fp32 accumulators in tensor memory.  Each
// operand value v is split three ways, hi = bf16(v), mid = bf16(v - hi), lo =
// bf16(v - hi - mid) (24 significant bits, as f32 has), and every 16-wide K
// step issues six products: hi*hi into one 128 x 256 accumulator, hi*mid,
// mid*hi, hi*lo, lo*hi and mid*mid into a second one (columns 256..511), the
// two added in f32 when the tile is stored; the dropped terms are below 2^-24
// of the product.  Measured on one tile of Q4_K-shaped weights against an
// fp64 product (K = 2560): 3.3e-6 relative, against 2.2e-6 for an f32 FMA
// loop, 5.4e-6 for a two-way split (hi, lo; three products) and 2.7e-3 for
// one bf16 product.  The two-way split's extra error, amplified through 32
// layers, put the 4B prefill's deep attention K/V rows past 1e-3 of the
// oracle's.
//
// Tiles.  A stage is a half-quarter: 32 inputs, one 64-byte row per matrix
// row, row r at r * 64, its 16-byte chunk c at (c ^ ((r >> 1) & 3)) * 16 (the
// 64-byte swizzle; the matrix descriptor's groups of 8 rows are 512 bytes
// apart).  A stage holds the weight tiles (hi, mid, lo: 8 KB each) and the
// input tiles of both token tiles ([hi | mid | lo] x [tile 0 | tile 1], 48 KB;
// a part's two token tiles are one 256-row operand); three 72 KB stages.  The
// inputs arrive already in this form: the kernels that produce a GEMM input
// write it as (half-quarter, 256-token pair) blocks (put_xt), and one bulk
// copy per stage brings a block in.  512 threads build the weight tiles:
// thread (row r = tid & 127, part = tid >> 7) dequantizes 16 weights of weight
// row r per quarter (the next quarter's raw bytes are loaded before this
// quarter's are decoded); parts 0, 1 fill a quarter's first half-quarter
// stage and parts 2, 3 its second, so the two builder groups fill alternate
// stages.  A 17th warp issues each stage's 12 MMAs.  A weight tile built once
// serves 256 tokens, and one instruction does 128 x 256 x 16.
constexpr int kMmaTile = 128 * 64;       // bytes of one 128 x 32 bf16 operand tile (64-byte rows)
constexpr int kMmaA = 3 * kMmaTile;      // a stage's weight tiles: hi, mid, lo
constexpr int kMmaB = 6 * kMmaTile;      // its input tiles: hi, mid, lo of two 128-token tiles ([part][tile])
constexpr int kMmaStage = kMmaA + kMmaB;  // one half-quarter (32 inputs) of a 128-row x 256-token tile
constexpr int kMmaStages = 3;
constexpr int kXtBytesPerValue = 6;      // a GEMM input value as put_xt tiles: hi, mid, lo
constexpr int kXtPairs = kPfChunk / 256;  // 256-token tile pairs of a chunk (input blocks per half-quarter)
constexpr int kMmaSmem = kMmaStages * kMmaStage + 1024 + 128;  // stages, 1024-byte alignment, barriers
constexpr int kMmaBuilders = 512;                               // 16 warps build the stages
constexpr int kMmaThreads = kMmaBuilders + 32;                  // + the warp that issues the MMAs
// kind::f16 instruction descriptor: f32 accumulator (bits 4-5 = 1), bf16 A and
// B (bits 7-9, 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t kMmaIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((256u >> 3) << 17) | ((128u >> 4) << 24);  // M 128, N 256
constexpr uint32_t kMmaIdescHalf = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);  // N 128

// Shared-memory matrix descriptor of a K-major tile with 64-byte rows and the
// 64-byte swizzle: start address >> 4, leading offset 16 B (unused by this
// layout), 8-row groups 512 B apart, descriptor version 1, swizzle mode 4 (64 B).
__device__ __forceinline__ uint64_t mma_sdesc(uint32_t addr) {
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(512 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(4) << 61);
}
__device__ __forceinline__ void mma_bf16(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// 16 consecutive accumulator columns of the warp's 32 lanes (wait::ld before use).
__device__ __forceinline__ void tmem_ld16(uint32_t ta, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(ta));
}
// The three-way split of one value: hi, mid, lo as bf16 (round to nearest).
__device__ __forceinline__ void bf16_split3(float v, __nv_bfloat16& h, __nv_bfloat16& m, __nv_bfloat16& l) {
    h = __float2bfloat16_rn(v);
    const float r = v - __bfloat162float(h);  // exact
    m = __float2bfloat16_rn(r);
    l = __float2bfloat16_rn(r - __bfloat162float(m));
}
// The three-way split of two values at once (one paired conversion per part),
// the same values bf16_split3 gives.
__device__ __forceinline__ void bf16x2_split3(float a, float b, uint32_t& h, uint32_t& m, uint32_t& l) {
    const __nv_bfloat162 hh = __floats2bfloat162_rn(a, b);
    const float ra = a - __low2float(hh), rb = b - __high2float(hh);  // exact
    const __nv_bfloat162 mm = __floats2bfloat162_rn(ra, rb);
    const __nv_bfloat162 ll = __floats2bfloat162_rn(ra - __low2float(mm), rb - __high2float(mm));
    h = *reinterpret_cast<const uint32_t*>(&hh);
    m = *reinterpret_cast<const uint32_t*>(&mm);
    l = *reinterpret_cast<const uint32_t*>(&ll);
}
// Row r of a 64-byte-row tile: its 16-byte chunk c (8 bf16) at
// r * 64 + (c ^ ((r >> 1) & 3)) * 16 (the 64-byte swizzle: byte-address bits
// 4-5 xor bits 7-8).
__device__ __forceinline__ int sw64(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }
// 16 values of row r (chunks c0, c0 + 1) into the hi, mid and lo tiles t0,
// t0 + kMmaTile, t0 + 2 kMmaTile.
__device__ __forceinline__ void put_row16(uint8_t* t0, int r, int c0, const float* v) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint32_t h[4], m[4], l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) bf16x2_split3(v[8 * c + 2 * i], v[8 * c + 2 * i + 1], h[i], m[i], l[i]);
        const int off = sw64(r, c0 + c);
        *reinterpret_cast<uint4*>(t0 + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(t0 + kMmaTile + off) = make_uint4(m[0], m[1], m[2], m[3]);
        *reinterpret_cast<uint4*>(t0 + 2 * kMmaTile + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}
// A GEMM input value (k, token p) of a prefill chunk in the tensor-core form:
// for half-quarter k / 32 and 256-token pair p / 256 one 48 KB block of six
// tiles [hi | mid | lo] x [tile 0 | tile 1] (128 tokens each), kXtPairs blocks
// per half-quarter; row p % 128, element k % 32.  Tokens P..kPfChunk-1 of a
// chunk are never stored.
__device__ __forceinline__ void put_xt(uint8_t* xt, int k, int p, float v) {
    uint8_t* t = xt + static_cast<size_t>((k >> 5) * kXtPairs + (p >> 8)) * kMmaB + ((p >> 7) & 1) * kMmaTile;
    const int row = p & 127;
    const int off = sw64(row, (k & 31) >> 3) + 2 * (k & 7);
    __nv_bfloat16 h, m, l;
    bf16_split3(v, h, m, l);
    *reinterpret_cast<__nv_bfloat16*>(t + off) = h;
    *reinterpret_cast<__nv_bfloat16*>(t + 2 * kMmaTile + off) = m;
    *reinterpret_cast<__nv_bfloat16*>(t + 4 * kMmaTile + off) = l;
}
// A GEMM input of a pass: k-major f32 [k][ld], or (ld == 0) the tiles of put_xt.
__device__ __forceinline__ void put_in(float* out, int ld, int k, int p, float v) {
    if (ld == 0) put_xt(reinterpret_cast<uint8_t*>(out), k, p, v);
    else out[static_cast<size_t>(k) * ld + p] = v;
}

// Y = W X over the quarters of split z (grid (ceil(n/128), ceil(P/128),
// splits), kMmaThreads threads, kMmaSmem bytes): W planar Q4_K / Q6_K [n x k]
// in the grouped layout, XT the inputs as put_xt tiles.  Output: split z at
// Y + z split_stride, token-major Y[t ldy + row] or, ROW_MAJOR, Y[row ldy + t]
// (k-major for a following GEMM).  err: a bounded wait that gave up sets
// DEVERR_FULL_WAIT and the CTA stores nothing.
//
// Warps 0..15 build stages (warp-level arrivals on `built`, no CTA barrier in
// the loop); warp 16 waits for a stage's `built` and `full` (its input tiles'
// bulk copy), issues its MMAs and commits them to `done`, which the builders
// wait on before they reuse the stage kMmaStages quarters later.
template <int QT, bool ROW_MAJOR>
__global__ void __launch_bounds__(kMmaThreads, 1) pf_mma_kernel(const uint8_t* __restrict__ W, int n, int k,
                                                                const uint8_t* __restrict__ XT, float* __restrict__ Y,
                                                                int ldy, size_t split_stride, int P, int q_per_split,
                                                                unsigned* __restrict__ err) {
    using Raw = typename std::conditional<QT == QT_Q6K, RawQ6, RawQ4>::type;
    extern __shared__ uint8_t mma_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mma_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* done = reinterpret_cast<uint64_t*>(sm + kMmaStages * kMmaStage);  // a stage's MMAs have completed
    uint64_t* full = done + kMmaStages;                                          // a stage's input tiles have landed
    uint64_t* built = full + kMmaStages;                                         // a stage's weight tiles are written
    uint32_t* tslot = reinterpret_cast<uint32_t*>(built + kMmaStages);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = blockIdx.x * 128, tok0 = blockIdx.y * 256;
    const int nb = k / 256, n8 = (n + 7) & ~7;
    const int q0 = blockIdx.z * q_per_split, q1 = min(4 * nb, q0 + q_per_split), nq = q1 - q0;
    const int nh = 2 * nq;  // half-quarter stages of the split
    if (tid == 0) {
        for (int i = 0; i < kMmaStages; ++i) {
            mbar_init(&done[i], 1);
            mbar_init(&full[i], 1);
            mbar_init(&built[i], kMmaBuilders / 64);  // the 8 warps of the half-quarter's builder group
        }
        fence_mbar_init();
    }
    if (warp == 0) {  // all 512 columns of tensor memory: two 128 x 256 f32 accumulators
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)), "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    }
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tslot;
    if (warp == kMmaBuilders / 32) {  // the MMA warp
        // a pair whose second token tile holds no token: 128-wide products
        const uint32_t idesc = tok0 + 128 < P ? kMmaIdesc : kMmaIdescHalf;
        if (lane == 0) {
            for (int h = 0, st = 0, use = 0; h < nh; ++h) {
                const bool ready = mbar_wait(&built[st], use & 1) && mbar_wait(&full[st], use & 1);
                if (ready) {
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t ah = smem_u32(sm + st * kMmaStage), am = ah + kMmaTile, al = ah + 2 * kMmaTile;
                    // B: the two token tiles of a part are one 256-row operand
                    const uint32_t bh = ah + kMmaA, bm = bh + 2 * kMmaTile, bl = bh + 4 * kMmaTile;
#pragma unroll
                    for (int s = 0; s < 2; ++s) {  // K steps of 16 (32 bytes into each 64-byte row)
                        const uint32_t o = 32 * s;
                        const uint32_t acc = (h > 0 || s > 0) ? 1u : 0u;
                        mma_bf16(tmem, mma_sdesc(ah + o), mma_sdesc(bh + o), idesc, acc);  // hi * hi
                        // the corrections, apart from hi * hi
                        mma_bf16(tmem + 256, mma_sdesc(ah + o), mma_sdesc(bm + o), idesc, acc);
                        mma_bf16(tmem + 256, mma_sdesc(am + o), mma_sdesc(bh + o), idesc, 1u);
                        mma_bf16(tmem + 256, mma_sdesc(ah + o), mma_sdesc(bl + o), idesc, 1u);
                        mma_bf16(tmem + 256, mma_sdesc(al + o), mma_sdesc(bh + o), idesc, 1u);
                        mma_bf16(tmem + 256, mma_sdesc(am + o), mma_sdesc(bm + o), idesc, 1u);
                    }
                } else {
                    atomicOr(err, static_cast<unsigned>(DEVERR_FULL_WAIT));
                }
                mma_commit(&done[st]);  // also when nothing was issued: the builders' waits stay matched
                if (++st == kMmaStages) {
                    st = 0;
                    ++use;
                }
            }
        }
        __syncwarp();
    } else {  // builders: thread (row r = tid & 127, part = tid >> 7), group part >> 1 builds half-quarter 2j + group
        const int r = tid & 127, part = tid >> 7, grp = part >> 1;
        const int grow = row0 + r;
        const bool row_ok = grow < n8;  // rows n..n8-1 are zero in the layout
        const int GB = QT == QT_Q6K ? 1680 : 1152;
        Raw cur{};
        if (nq > 0 && row_ok) raw_load(W + grouped_offset(n8, nb, grow >> 3, q0 >> 2, GB), grow & 7, q0 & 3, part, cur);
        bool failed = false;
        for (int j = 0; j < nq; ++j) {
            const int qi = q0 + j, h = 2 * j + grp, st = h % kMmaStages, use = h / kMmaStages;
            uint8_t* sb = sm + st * kMmaStage;
            const bool free = use == 0 || mbar_wait(&done[st], (use - 1) & 1);  // the MMAs that read this stage are done
            if (free) {
                if ((tid & 255) == 0) {  // the half-quarter's input tiles of the CTA's two token tiles
                    mbar_arrive_expect_tx(&full[st], kMmaB);
                    bulk_g2s(sb + kMmaA, XT + static_cast<size_t>((2 * qi + grp) * kXtPairs + blockIdx.y) * kMmaB, kMmaB,
                             &full[st], policy_evict_first());
                }
                Raw nxt{};  // the next quarter's raw bytes, in flight while this one is decoded
                if (qi + 1 < q1 && row_ok)
                    raw_load(W + grouped_offset(n8, nb, grow >> 3, (qi + 1) >> 2, GB), grow & 7, (qi + 1) & 3, part,
                             nxt);
                float v[16];
                if (row_ok) {
                    raw_decode(cur, qi & 3, part, v);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
                }
                put_row16(sb, r, 2 * (part & 1), v);
                cur = nxt;
            } else {
                failed = true;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the tiles, visible to the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&built[st]);
        }
        if (failed) atomicOr(err, static_cast<unsigned>(DEVERR_FULL_WAIT));
    }
    bool ok = nh == 0 || mbar_wait(&done[(nh - 1) % kMmaStages], ((nh - 1) / kMmaStages) & 1);  // all MMAs done
    ok = __syncthreads_and(ok && !__ldcg(err)) != 0;  // uniform: the accumulator loads are warp-collective
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (ok && warp < kMmaBuilders / 32) {  // warp w: accumulator lanes 32 (w & 3) .., token columns 64 (w >> 2) ..
        const int lq = warp & 3, cb = 64 * (warp >> 2);
        const int row = row0 + 32 * lq + lane;
        float* Yz = Y + blockIdx.z * split_stride;
#pragma unroll 1
        for (int c = 0; c < 64; c += 16) {
            const int tc = cb + c;  // the CTA's token column: tile tc >> 7, column tc & 127
            float v[16];
            if (nq > 0) {
                const uint32_t ta = tmem + (static_cast<uint32_t>(32 * lq) << 16) + static_cast<uint32_t>(tc);
                uint32_t hi[16], lo[16];
                tmem_ld16(ta, hi);        // hi * hi, columns 0..255
                tmem_ld16(ta + 256, lo);  // the corrections, columns 256..511
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(hi[i]) + __uint_as_float(lo[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.0f;
            }
            if (row < n) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int t = tok0 + tc + i;
                    if (t < P) {
                        if (ROW_MAJOR) Yz[static_cast<size_t>(row) * ldy + t] = v[i];
                        else Yz[static_cast<size_t>(t) * ldy + row] = v[i];
                    }
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
}

// ------------------------------------ small-batch GEMV on the engine's pipeline
// Y = W X for at most 4 columns (a lockstep decode step of up to 4
// sequences), W in the engine's grouped, slice-major layout and read once for
// all columns; X packed [k][4] (the 4 columns of one k are one float4).
//
// Work split.  The (K slice, 8-row group) tasks, slice-major and weighted by
// the slice width, are cut into one contiguous range per CTA (two CTAs per
// SM).  A task writes its rows' sums over its slice to output part s (s the
// slice index) and the consumer of Y adds the parts in slice order, so a CTA
// stages the inputs of one slice (two at a range's seam) once, and its
// producer warp streams the CTA's rows of that slice into the engine's ring
// of shared-memory stages (one bulk copy per stage of up to PP row passes).
//
// Arithmetic.  In a slice of G = 2^lg chunks of 64 weights, G lanes cover one
// row (the engine's lane partition), lane j its chunk; a lane takes all the
// passes of a stage together, so every input float4 it reads serves each of
// them.  A 4- or 6-bit code c becomes the float 1 + c 2^-e by a shift that
// puts it into the mantissa of 1.0 and one mask-or, so a lane's sum over a
// sub-block is sum x + 2^-e sum c x: the plain sum of x over the sub-block
// (formed once per slice and shared by every lane) is taken off and the rest
// scaled by 2^e, both exact.  The products keep f32 rounding (2^-24 of
// sum |x| per sub-block, times 2^e <= 2^8 after the subtraction).  The integer
// scales and the Q4_K minimum enter once per sub-block, as the GGUF formulas
// have them, and a transposed xor tree sums the 4 columns over a row's G
// lanes (lane j ends with column j >> (lg - 2)).
constexpr int kBmSliceK = 2048;  // inputs staged per slice (the widest slice: 32 chunks of 64)
template <int QT>
struct BmPasses {
    static constexpr int value = QT == QT_Q4K ? 3 : 2;  // row passes per stage (27 KB / 26 KB)
};
constexpr int kBmXs = kBmSliceK + kBmSliceK / 64 + kBmSliceK / 512;  // staged float4 slots (with the padding)
constexpr int kBmXsum = kBmSliceK / 16 + kBmSliceK / 256;           // sub-block sum slots (with the padding)

// Slot of input k in the staged slice: a row's lanes read inputs 64 (Q4_K) or
// 256 (Q6_K) apart at the same time, which would fall on the same banks; one
// float4 of padding after every 64 and one more after every 512 puts the 8
// lanes of a shared-memory phase on 8 different 16-byte bank groups.  A run
// of 64 inputs from a multiple of 64 stays contiguous, so a lane reads its
// chunk at fixed offsets from one pointer.
__device__ __forceinline__ int xs_at(int k) { return k + (k >> 6) + (k >> 9); }
// Slot of sub-block sum i (of 32 inputs for Q4_K, 16 for Q6_K): the lanes of a
// phase read sums 2 (Q4_K) or 16 (Q6_K) apart; one float4 of padding after
// every 8 (Q4_K) or 16 (Q6_K) puts them on different bank groups.
template <int QT>
__device__ __forceinline__ int xsum_at(int i) { return QT == QT_Q4K ? i + (i >> 3) : i + (i >> 4); }

// a += q x, as two packed f32x2 multiply-adds (each half rounds as fmaf does)
__device__ __forceinline__ void fma4(float4& a, float q, const float4& x) {
    const float2 qq = make_float2(q, q);
    const float2 lo = __ffma2_rn(qq, make_float2(x.x, x.y), make_float2(a.x, a.y));
    const float2 hi = __ffma2_rn(qq, make_float2(x.z, x.w), make_float2(a.z, a.w));
    a = make_float4(lo.x, lo.y, hi.x, hi.y);
}
// Byte b of v moved to bits 15..22 (Q4_K: low nibble at 15, high at 19) or
// 17..22 (Q6_K codes), the mantissa bits of 1.0 that the mask-or fills.
template <int B, int AT>
__device__ __forceinline__ unsigned byte_to(unsigned v) {
    constexpr int sh = AT - 8 * B;
    return sh >= 0 ? v << sh : v >> -sh;
}
__device__ __forceinline__ float one_plus(unsigned t, unsigned mask) { return __uint_as_float((t & mask) | 0x3F800000u); }

// The 4 columns of v summed over the G = 2^lg lanes of the lane's row: lane j
// of the row returns column j >> (lg - 2) (a transposed xor tree: two
// exchanges halve the columns, the rest is a plain tree).
__device__ __forceinline__ float row_sum4(const float4& v, int lg, int lane) {
    const int o1 = 1 << (lg - 1), o2 = 1 << (lg - 2);
    const bool b1 = lane & o1, b2 = lane & o2;
    float a0 = b1 ? v.z : v.x, a1 = b1 ? v.w : v.y;
    a0 += __shfl_xor_sync(FULL, b1 ? v.x : v.z, o1);
    a1 += __shfl_xor_sync(FULL, b1 ? v.y : v.w, o1);
    float r = b2 ? a1 : a0;
    r += __shfl_xor_sync(FULL, b2 ? a0 : a1, o2);
    for (int o = o2 >> 1; o > 0; o >>= 1) r += __shfl_xor_sync(FULL, r, o);
    return r;
}

// What a lane needs of its row and chunk in one slice.
struct BmLane {
    int lg, rl, j, q;
    int o0, o1, o2;  // Q4_K: the row's block; Q6_K: [A | B | H] record, scale record, d (as LaneRow)
    int k0;          // the chunk's first input, relative to the slice
    int col;         // the column this lane stores
    bool store;
};
template <int QT>
__device__ __forceinline__ BmLane bm_lane(int lg, int warp, int lane, int nm) {
    BmLane L;
    L.lg = lg;
    const int rpw = 32 >> lg, kbl = (1 << lg) >> 2;
    L.rl = warp * rpw + (lane >> lg);
    L.j = lane & ((1 << lg) - 1);
    int bl;
    lane_chunk<QT>(L.j, lg, bl, L.q);
    if constexpr (QT == QT_Q4K) {
        L.o0 = ((L.rl >> 3) * kbl + bl) * group_block_bytes(QT) + (L.rl & 7) * 144;
        L.o1 = L.o2 = 0;
        L.k0 = 256 * bl + 64 * L.q;
    } else {
        const int base = ((L.rl >> 3) * kbl + bl) * group_block_bytes(QT), rr = L.rl & 7, u = 4 * rr + L.q;
        L.o0 = base + 48 * u;
        L.o1 = base + 1536 + 4 * u;
        L.o2 = base + 1664 + 2 * rr;
        L.k0 = 256 * bl + 128 * (L.q >> 1) + 16 * (L.q & 1);
    }
    L.col = L.j >> (lg - 2);
    L.store = (L.j & ((1 << (lg - 2)) - 1)) == 0 && L.col < nm;
    return L;
}

// Where a row's slice sums go: output part Yp (token-major Y[t][ldy] or,
// ROW_MAJOR, Y[row][ldy]), or (AM, the argmax mode) the CTA's row sums ys
// [row - r0][4] in shared memory, added over the slices in slice order.
struct BmOut {
    float* Yp;
    int ldy;
    float* ys;
    int r0;
    bool first;
};
template <bool ROW_MAJOR, bool AM>
__device__ __forceinline__ void bm_put(const BmLane& L, float v, int row, int rb, const BmOut& o) {
    if (L.store && row < rb) {
        if (AM) {
            float* y = o.ys + 4 * (row - o.r0) + L.col;
            *y = o.first ? v : *y + v;
        } else if (ROW_MAJOR) {
            o.Yp[static_cast<size_t>(row) * o.ldy + L.col] = v;
        } else {
            o.Yp[static_cast<size_t>(L.col) * o.ldy + row] = v;
        }
    }
}

// NP Q4_K row passes of a stage (the first at ps), rows row, row + U, ...
template <int NP, bool ROW_MAJOR, bool AM>
__device__ void bm_q4_passes(const BmLane& L, const uint8_t* ps, const float4* xs, const float4* xsum, int row, int U,
                             int rb, const BmOut& o) {
    constexpr int PB = kStageBlockRows * 144;
    float4 s0[NP], s1[NP];
#pragma unroll
    for (int t = 0; t < NP; ++t) {
        s0[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        s1[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float4* xc = xs + xs_at(L.k0);  // the chunk's 64 inputs, contiguous
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {  // bytes 16h .. 16h + 15 of the chunk's 32
        uint4 cw[NP];
#pragma unroll
        for (int t = 0; t < NP; ++t) cw[t] = *reinterpret_cast<const uint4*>(ps + t * PB + L.o0 + 16 + 32 * L.q + 16 * h);
        const float4* xb = xc + 16 * h;
#pragma unroll
        for (int i = 0; i < 16; ++i) {  // byte i: low nibble -> input k0 + 16h + i, high -> k0 + 32 + 16h + i
            const float4 xl = xb[i], xh = xb[32 + i];
#pragma unroll
            for (int t = 0; t < NP; ++t) {
                unsigned v = u4w(cw[t], i >> 2);
                switch (i & 3) {
                    case 0: v = byte_to<0, 15>(v); break;
                    case 1: v = byte_to<1, 15>(v); break;
                    case 2: v = byte_to<2, 15>(v); break;
                    default: v = byte_to<3, 15>(v); break;
                }
                fma4(s0[t], one_plus(v, 0x00078000u), xl);  // 1 + q / 256
                fma4(s1[t], one_plus(v, 0x00780000u), xh);  // 1 + q / 16
            }
        }
    }
    const float4 X0 = xsum[xsum_at<QT_Q4K>(L.k0 >> 5)], X1 = xsum[xsum_at<QT_Q4K>((L.k0 >> 5) + 1)];
#pragma unroll
    for (int t = 0; t < NP; ++t) {
        const uint4 hdr = *reinterpret_cast<const uint4*>(ps + t * PB + L.o0);
        const float d = f16_to_f32(static_cast<uint16_t>(hdr.x & 0xffffu));
        const float dmin = f16_to_f32(static_cast<uint16_t>(hdr.x >> 16));
        // 6-bit scale / min of sub-blocks 2q (low nibbles) and 2q + 1 (high), as dot_q4k takes them
        int sc[2], mn[2];
        const bool low = L.q < 2;
        const unsigned asc = low ? hdr.y : hdr.w, amn = low ? hdr.z : hdr.w;
        const unsigned msk = low ? 63u : 15u, mhi = low ? 0u : 0x30u, sm4 = low ? 0u : 4u;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const unsigned sh8 = 16u * static_cast<unsigned>(L.q & 1) + 8u * u;
            sc[u] = static_cast<int>(((asc >> sh8) & msk) | ((hdr.y >> (sh8 + 2u)) & mhi));
            mn[u] = static_cast<int>(((amn >> (sh8 + sm4)) & msk) | ((hdr.z >> (sh8 + 2u)) & mhi));
        }
        const float a0 = 256.0f * d * static_cast<float>(sc[0]), a1 = 16.0f * d * static_cast<float>(sc[1]);
        const float b0 = dmin * static_cast<float>(mn[0]), b1 = dmin * static_cast<float>(mn[1]);
        float4 acc;
        acc.x = fmaf(a0, s0[t].x - X0.x, fmaf(a1, s1[t].x - X1.x, -fmaf(b0, X0.x, b1 * X1.x)));
        acc.y = fmaf(a0, s0[t].y - X0.y, fmaf(a1, s1[t].y - X1.y, -fmaf(b0, X0.y, b1 * X1.y)));
        acc.z = fmaf(a0, s0[t].z - X0.z, fmaf(a1, s1[t].z - X1.z, -fmaf(b0, X0.z, b1 * X1.z)));
        acc.w = fmaf(a0, s0[t].w - X0.w, fmaf(a1, s1[t].w - X1.w, -fmaf(b0, X0.w, b1 * X1.w)));
        bm_put<ROW_MAJOR, AM>(L, row_sum4(acc, L.lg, L.j), row + t * U, rb, o);
    }
}

// NP Q6_K row passes (planar records): per 16-weight group s4 with int8 scale
// sc, sc * (sum (c - 32) x) = sc * (64 (sum (1 + c/64) x - X) - 32 X), then d.
template <int NP, bool ROW_MAJOR, bool AM>
__device__ void bm_q6_passes(const BmLane& L, const uint8_t* ps, const float4* xs, const float4* xsum, int row, int U,
                             int rb, const BmOut& o) {
    constexpr int PB = kStageBlockRows * 210;
    uint4 A[NP], B[NP], H[NP];
    unsigned S[NP];
    float4 acc[NP];
#pragma unroll
    for (int t = 0; t < NP; ++t) {
        const uint8_t* rec = ps + t * PB + L.o0;
        A[t] = *reinterpret_cast<const uint4*>(rec);
        B[t] = *reinterpret_cast<const uint4*>(rec + 16);
        H[t] = *reinterpret_cast<const uint4*>(rec + 32);
        S[t] = *reinterpret_cast<const unsigned*>(ps + t * PB + L.o1);
        acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4) {  // group s4: inputs k0 + 32 s4 .. + 15
        const int kk = L.k0 + 32 * s4;
        const float4* xg = xs + xs_at(kk);  // the group's 16 inputs, contiguous
        float4 sg[NP];
#pragma unroll
        for (int t = 0; t < NP; ++t) sg[t] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            unsigned c4[NP];  // the 4 codes of inputs 4w .. 4w + 3 of the group (dot_q6k's unpacking)
#pragma unroll
            for (int t = 0; t < NP; ++t) {
                const unsigned a = u4w(A[t], w), bb = u4w(B[t], w), hh = u4w(H[t], w);
                if (s4 == 0) c4[t] = (a & 0x0f0f0f0fu) | ((hh << 4) & 0x30303030u);
                else if (s4 == 1) c4[t] = (bb & 0x0f0f0f0fu) | ((hh << 2) & 0x30303030u);
                else if (s4 == 2) c4[t] = ((a >> 4) & 0x0f0f0f0fu) | (hh & 0x30303030u);
                else c4[t] = ((bb >> 4) & 0x0f0f0f0fu) | ((hh >> 2) & 0x30303030u);
            }
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int i = 4 * w + b;
                const float4 x = xg[i];
#pragma unroll
                for (int t = 0; t < NP; ++t) {
                    unsigned v;
                    switch (b) {
                        case 0: v = byte_to<0, 17>(c4[t]); break;
                        case 1: v = byte_to<1, 17>(c4[t]); break;
                        case 2: v = byte_to<2, 17>(c4[t]); break;
                        default: v = byte_to<3, 17>(c4[t]); break;
                    }
                    fma4(sg[t], one_plus(v, 0x007E0000u), x);  // 1 + c / 64
                }
            }
        }
        const float4 X = xsum[xsum_at<QT_Q6K>(kk >> 4)];
        const float4 m32 = make_float4(-32.0f * X.x, -32.0f * X.y, -32.0f * X.z, -32.0f * X.w);
#pragma unroll
        for (int t = 0; t < NP; ++t) {
            const float sc = static_cast<float>(static_cast<int>(S[t] << (24 - 8 * s4)) >> 24);
            acc[t].x = fmaf(sc, fmaf(64.0f, sg[t].x - X.x, m32.x), acc[t].x);
            acc[t].y = fmaf(sc, fmaf(64.0f, sg[t].y - X.y, m32.y), acc[t].y);
            acc[t].z = fmaf(sc, fmaf(64.0f, sg[t].z - X.z, m32.z), acc[t].z);
            acc[t].w = fmaf(sc, fmaf(64.0f, sg[t].w - X.w, m32.w), acc[t].w);
        }
    }
#pragma unroll
    for (int t = 0; t < NP; ++t) {
        const float d = f16_to_f32(*reinterpret_cast<const uint16_t*>(ps + t * PB + L.o2));
        const float4 v = make_float4(d * acc[t].x, d * acc[t].y, d * acc[t].z, d * acc[t].w);
        bm_put<ROW_MAJOR, AM>(L, row_sum4(v, L.lg, L.j), row + t * U, rb, o);
    }
}

// Rows [ra, rb) of one slice (2^lg lanes per row), stage by stage.
template <int QT, bool ROW_MAJOR, bool AM>
__device__ void bm4_slice(Pipe& p, int lg, int ra, int rb, const float4* xs, const float4* xsum, const BmOut& o, int nm,
                          int warp, int lane) {
    constexpr int PP = BmPasses<QT>::value;
    constexpr int PB = kStageBlockRows * block_bytes(QT);
    const BmLane L = bm_lane<QT>(lg, warp, lane, nm);
    const int U = 8 * (32 >> lg);
    for (int row0 = ra; row0 < rb; row0 += U * PP) {
        const int npass = min(PP, (rb - row0 + U - 1) / U);  // uniform over the CTA
        p.wait_full();
        const uint8_t* ps = p.cur();
        const int row = row0 + L.rl;
        if constexpr (QT == QT_Q4K) {
            if (npass == 3) bm_q4_passes<3, ROW_MAJOR, AM>(L, ps, xs, xsum, row, U, rb, o);
            else if (npass == 2) bm_q4_passes<2, ROW_MAJOR, AM>(L, ps, xs, xsum, row, U, rb, o);
            else bm_q4_passes<1, ROW_MAJOR, AM>(L, ps, xs, xsum, row, U, rb, o);
        } else {
            if (npass == 2) bm_q6_passes<2, ROW_MAJOR, AM>(L, ps, xs, xsum, row, U, rb, o);
            else bm_q6_passes<1, ROW_MAJOR, AM>(L, ps, xs, xsum, row, U, rb, o);
        }
        p.release();
    }
}

// First task (slice-major index s * units + g) that starts at or after weight
// position pos, a task of slice s weighing 2^lg_s.
__device__ int bm_task_at(const GemvShape& sh, long long pos) {
    long long c = 0;
    for (int s = 0; s < sh.nsl; ++s) {
        const int lg = sh.sl_lg[s];
        const long long span = static_cast<long long>(sh.units) << lg;
        if (pos < c + span) return s * sh.units + static_cast<int>((pos - c + (1LL << lg) - 1) >> lg);
        c += span;
    }
    return sh.nsl * sh.units;
}

// The CTA's work as a walk over (slice s, rows [ra, rb)) segments.  Parts
// mode: its range of tasks, a run of consecutive groups of one slice per
// segment.  AM: its own rows (whole 8-row groups) in every slice, slice by slice.
template <bool AM>
struct BmWalk {
    int it, end, r0, r1;
    __device__ explicit BmWalk(const GemvShape& sh) {
        if (AM) {
            cta_rows(sh.units, sh.n, r0, r1);
            it = 0;
            end = sh.nsl;
        } else {
            long long tot = 0;
            for (int s = 0; s < sh.nsl; ++s) tot += static_cast<long long>(sh.units) << sh.sl_lg[s];
            it = bm_task_at(sh, tot * blockIdx.x / gridDim.x);
            end = bm_task_at(sh, tot * (blockIdx.x + 1) / gridDim.x);
            r0 = r1 = 0;
        }
    }
    __device__ bool next(const GemvShape& sh, int& s, int& ra, int& rb) {
        if (it >= end) return false;
        if (AM) {
            s = it++;
            ra = r0;
            rb = r1;
        } else {
            s = it / sh.units;
            const int g = it - s * sh.units, ge = min(sh.units, g + (end - it));
            ra = 8 * g;
            rb = min(8 * ge, sh.n);
            it += ge - g;
        }
        return true;
    }
};

// The producer warp: the CTA's segments in order, each in stages of PP passes
// (one contiguous piece of the grouped layout per stage).
template <int QT, bool AM>
__device__ bool bm_produce(Pipe& p, const GemvShape& sh) {
    constexpr int GB = group_block_bytes(QT), PP = BmPasses<QT>::value;
    BmWalk<AM> wk(sh);
    int s, ra, rb;
    while (wk.next(sh, s, ra, rb)) {
        const int lg = sh.sl_lg[s], kbl = (1 << lg) >> 2, U = 8 * (32 >> lg) * PP, b0 = sh.sl_c0[s] >> 2;
        for (int row0 = ra; row0 < rb; row0 += U) {
            const int rows = min(U, rb - row0);
            if (!p.acquire()) return false;
            const unsigned bytes = static_cast<unsigned>((rows + 7) >> 3) * kbl * GB;
            p.expect(bytes);
            if (p.lane == 0)
                p.copy(p.cur(), sh.w0 + (static_cast<size_t>(sh.n8 / 8) * b0 + static_cast<size_t>(row0 >> 3) * kbl) * GB,
                       bytes);
            p.commit();
        }
    }
    return true;
}

// Per column c < nm of the argmax mode: the sequence's first-index argmax
// word (two u64: key, arrival count; zero between launches), its token slots
// (slots[0] = token, slots[2] = token | bit 31 when an error word is set), its
// allow bitset and error word.
struct BmArgmax {
    unsigned long long* ws[4];
    int* slots[4];
    const uint32_t* allow[4];
    const unsigned* err[4];
};

// Parts mode: output part s (slice s) at Y + s * split_stride, Y[t][ldy]
// (token-major) or, ROW_MAJOR, Y[row][ldy]; columns >= nm are not stored.
// AM: the rows' full sums stay in shared memory (ys at ys_off) and each column
// ends in a masked first-index argmax over all rows (the lm_head of up to 4
// sequences: EpiArgmaxStep's key and last-arriver protocol per column).
template <int QT, bool ROW_MAJOR, bool AM>
__global__ void __launch_bounds__(kThreads, 2) bm4_kernel(const GemvShape sh, const float* X, int xq,
                                                          float* Y, int ldy, size_t split_stride, int nm,
                                                          int ring_off, const BmArgmax am) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    float4* xs = reinterpret_cast<float4*>(smem + 16 * kMaxStages);  // [kBmXs]
    float4* xsum = xs + kBmXs;                                        // [kBmXsum]: sums of 32 (Q4_K) or 16 inputs
    float* ys = reinterpret_cast<float*>(xsum + kBmXsum);            // AM: [rows_cta][4]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();
    if (tid == 0) {
        for (int st = 0; st < sh.stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    Pipe p{full, empty, smem + ring_off, sh.stages, BmPasses<QT>::value * stage_bytes_of(QT), 0u, sh.err, sh.err, lane,
           0ull};
    if (warp == kConsumerWarps) {  // the weights depend on no earlier kernel: they stream in before the wait
        p.pol = policy_evict_first();
        if (!bm_produce<QT, AM>(p, sh)) p.drain();
        return;
    }
    pdl_wait();  // X (and the output parts this launch overwrites) belong to the earlier kernels
    const float4* X4 = reinterpret_cast<const float4*>(X);
    constexpr int SL = QT == QT_Q4K ? 32 : 16;  // inputs per sub-block sum
    BmWalk<AM> wk(sh);
    int s, ra, rb;
    while (wk.next(sh, s, ra, rb)) {
        const int lg = sh.sl_lg[s], kn = 64 << lg, kb = 64 * sh.sl_c0[s];
        // the slice's inputs, four loads in flight per thread (kn is a multiple of kConsumers)
        for (int i0 = 0; i0 < kn; i0 += 4 * kConsumers) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (i0 + u * kConsumers < kn) v[u] = __ldcg(X4 + static_cast<size_t>(kb + i0 + u * kConsumers + tid) * xq);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (i0 + u * kConsumers < kn) xs[xs_at(i0 + u * kConsumers + tid)] = v[u];
        }
        bar_sync(1, kConsumers);
        for (int e = tid; e < 4 * (kn / SL); e += kConsumers) {  // (sub-block, column) sums
            const int sb = e >> 2, c = e & 3;
            float a = 0.0f;
#pragma unroll 8
            for (int i = 0; i < SL; ++i) a += reinterpret_cast<const float*>(xs + xs_at(SL * sb + i))[c];
            reinterpret_cast<float*>(xsum + xsum_at<QT>(sb))[c] = a;
        }
        bar_sync(1, kConsumers);
        const BmOut o{Y + s * split_stride, ldy, ys, wk.r0, s == 0};
        bm4_slice<QT, ROW_MAJOR, AM>(p, lg, ra, rb, xs, xsum, o, nm, warp, lane);
        bar_sync(1, kConsumers);  // xs, xsum (and AM: the slice's row sums) are complete
    }
    if constexpr (AM) {
        unsigned long long best[4] = {0ull, 0ull, 0ull, 0ull};
        for (int r = wk.r0 + tid; r < wk.r1; r += kConsumers) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (c < nm) {
                    const bool ok = (__ldcg(am.allow[c] + (r >> 5)) >> (r & 31)) & 1u;
                    const unsigned long long key =
                        argmax_key(ok ? ys[4 * (r - wk.r0) + c] : -FLT_MAX, static_cast<unsigned>(r));
                    best[c] = key > best[c] ? key : best[c];
                }
            }
        }
        unsigned long long* red = reinterpret_cast<unsigned long long*>(xsum);  // [warp][4]
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            best[c] = warp_max_u64(best[c]);
            if (lane == 0) red[4 * warp + c] = best[c];
        }
        bar_sync(1, kConsumers);
        if (tid < nm) {
            const int c = tid;
            unsigned long long m = 0ull;
            for (int w = 0; w < kConsumerWarps; ++w) m = red[4 * w + c] > m ? red[4 * w + c] : m;
            atomicMax(am.ws[c], m);
            __threadfence();
            const unsigned prev = atomicAdd(reinterpret_cast<unsigned*>(am.ws[c] + 1), 1u);
            if (prev == gridDim.x - 1) {  // the last CTA for this column publishes
                __threadfence();
                const unsigned long long key = atomicExch(am.ws[c], 0ull);
                atomicExch(reinterpret_cast<unsigned*>(am.ws[c] + 1), 0u);
                const unsigned tok = key ? argmax_key_index(key) : 0u;
                const unsigned e = __ldcg(am.err[c]) | __ldcg(sh.err);
                am.slots[c][0] = static_cast<int>(tok);
                am.slots[c][2] = static_cast<int>(tok | (e ? 0x80000000u : 0u));
            }
        }
    }
}

// Launch of bm4_kernel over nm <= 4 columns: input k of the group is the
// float4 at X + k * xq floats (xq = 4: packed [k][4]; 8: one half of packed
// [k][8]).  Parts mode: *parts = the K slices (output parts, split_stride
// apart).  AM: the argmax words of am.  err: the device error word of the
// bounded ring waits.
template <int QT, bool ROW_MAJOR, bool AM>
int launch_bm4(const uint8_t* W, int n, int k, const float* X, int xq, float* Y, int ldy, size_t split_stride, int nm,
               const BmArgmax& am, unsigned* err, cudaStream_t st, int* parts) {
    if (!err) return set_err(QG_ERR_CUDA, "small-batch GEMV: no device error word");
    if (nm < 1 || nm > 4) return set_err(QG_ERR_SHAPE, "small-batch GEMV: %d columns (served: 1..4)", nm);
    constexpr int PP = BmPasses<QT>::value;
    int grid = 1;
    GemvShape sh = gemv_geometry(QT, false, W, nullptr, n, k, 0, 0, err, &grid, PP);  // AM: whole row groups per CTA
    if (sh.nsl > kPfMaxSplit) return set_err(QG_ERR_SHAPE, "small-batch GEMV: k = %d has %d slices", k, sh.nsl);
    sh.pp = PP;
    if (!AM) grid = static_cast<int>(std::min<long long>(2LL * device_sms(), static_cast<long long>(sh.units) * sh.nsl));
    const int ys_bytes = AM ? 16 * sh.rows_cta : 0;
    const int ring_off = (16 * kMaxStages + 16 * kBmXs + 16 * kBmXsum + ys_bytes + 127) & ~127;
    const int slot = PP * stage_bytes_of(QT);
    int stages = (kCtaSmemBytes - ring_off) / slot;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return set_err(QG_ERR_SHAPE, "small-batch GEMV: %d x %d leaves no ring in shared memory", n, k);
    sh.stages = stages;
    const int smem = ring_off + stages * slot;
    auto kern = bm4_kernel<QT, ROW_MAJOR, AM>;
    if (int rc = grant_smem(reinterpret_cast<const void*>(kern), smem)) return rc;
    if (int e_ = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, true, sh, X, xq / 4, Y, ldy, split_stride, nm,
                            ring_off, am))
        return e_;
    if (parts) *parts = sh.nsl;
    return QG_OK;
}

// Z = the `parts` split sums of a projection, added in split order.
__global__ void pf_sum_parts_kernel(const float* Yp, int parts, size_t stride, float* Z,
                                    size_t count) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= count) return;
    float v = Yp[i];
    for (int z0 = 1; z0 < parts; z0 += 4) {  // four parts' loads in flight, added in part order
        float t[4];
#pragma unroll
        for (int zz = 0; zz < 4; ++zz) t[zz] = z0 + zz < parts ? Yp[(z0 + zz) * stride + i] : 0.0f;
#pragma unroll
        for (int zz = 0; zz < 4; ++zz)
            if (z0 + zz < parts) v += t[zz];
    }
    Z[i] = v;
}

// X[p] = E[tok[p]].  Grid P.
__global__ void pf_embed_kernel(const float* E, const int* tok, int H, float* X) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    const int p = blockIdx.x;
    const float* src = E + static_cast<size_t>(tok[p]) * H;
    for (int i = threadIdx.x; i < H; i += blockDim.x) X[static_cast<size_t>(p) * H + i] = src[i];
}

// Per column of a batched decode pass, where the final residual stream is
// also stored (each sequence's state), or null.
struct HOut {
    float* h[kMaxSeg];
};

// X[p] += the `parts` split sums (in split order); then, when w is given,
// RMSNorm(X[p]) * w into column p of the GEMM input Xn (put_in); with ho.h[p],
// X[p] is also stored there.  Grid P.  SMALL (a batched decode step, P <= 16):
// 1024 threads, each holding the elements tid + 1024 e (H <= 16384), every
// load issued before the first sum needs one; else (a prefill chunk) 256
// threads striding over H, so that all P CTAs are resident at once.
constexpr int kAddNormWide = 1024, kAddNormPer = 16;
template <bool SMALL, int PER = 1>  // PER: values per thread of the wide variant (H <= 1024 PER)
__global__ void __launch_bounds__(SMALL ? kAddNormWide : 256)
    pf_add_norm_kernel(float* X, const float* Yp, int parts, size_t split_stride,
                       const float* w, float* Xn, int ldn, int H, float eps, const HOut ho) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    constexpr int T = SMALL ? kAddNormWide : 256;
    __shared__ float red[T / 32];
    const int p = blockIdx.x, tid = threadIdx.x;
    float* x = X + static_cast<size_t>(p) * H;
    const float* yp = Yp + static_cast<size_t>(p) * H;
    float* hp = p < kMaxSeg ? ho.h[p] : nullptr;
    float ss = 0.0f;
    float v[SMALL ? PER : 1];
    if constexpr (SMALL) {
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int i = tid + T * e;
            v[e] = i < H ? x[i] : 0.0f;
        }
        if (parts > 0) {
            float y[PER];
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                const int i = tid + T * e;
                y[e] = i < H ? yp[i] : 0.0f;
            }
            constexpr int D = PER <= 4 ? 4 : 1;  // parts whose loads are in flight together (registers allowing)
            if constexpr (D == 1) {
                for (int z = 1; z < parts; ++z)
#pragma unroll
                    for (int e = 0; e < PER; ++e) {
                        const int i = tid + T * e;
                        if (i < H) y[e] += yp[z * split_stride + i];
                    }
            } else {
                for (int z0 = 1; z0 < parts; z0 += D) {  // added in part order
                    float tz[D][PER];
#pragma unroll
                    for (int zz = 0; zz < D; ++zz)
#pragma unroll
                        for (int e = 0; e < PER; ++e) {
                            const int i = tid + T * e;
                            tz[zz][e] = (z0 + zz < parts && i < H) ? yp[(z0 + zz) * split_stride + i] : 0.0f;
                        }
#pragma unroll
                    for (int zz = 0; zz < D; ++zz)
#pragma unroll
                        for (int e = 0; e < PER; ++e)
                            if (z0 + zz < parts) y[e] += tz[zz][e];
                }
            }
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                const int i = tid + T * e;
                if (i < H) {
                    v[e] += y[e];
                    x[i] = v[e];
                }
            }
        }
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int i = tid + T * e;
            if (i < H) {
                ss = fmaf(v[e], v[e], ss);
                if (hp) hp[i] = v[e];
            }
        }
    } else {
        for (int i = tid; i < H; i += T) {
            float u = x[i];
            if (parts > 0) {
                float y = yp[i];
                for (int z0 = 1; z0 < parts; z0 += 4) {  // four parts' loads in flight, added in part order
                    float t4[4];
#pragma unroll
                    for (int zz = 0; zz < 4; ++zz) t4[zz] = z0 + zz < parts ? yp[(z0 + zz) * split_stride + i] : 0.0f;
#pragma unroll
                    for (int zz = 0; zz < 4; ++zz)
                        if (z0 + zz < parts) y += t4[zz];
                }
                u += y;
                x[i] = u;
            }
            if (hp) hp[i] = u;
            ss = fmaf(u, u, ss);
        }
    }
    if (!w) return;
    ss = warp_sum(ss);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    float t = 0.0f;
#pragma unroll
    for (int i = 0; i < T / 32; ++i) t += red[i];
    const float r = 1.0f / sqrtf(t / static_cast<float>(H) + eps);
    if constexpr (SMALL) {
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int i = tid + T * e;
            if (i < H) put_in(Xn, ldn, i, p, (v[e] * r) * w[i]);
        }
    } else {
        for (int i = tid; i < H; i += T) put_in(Xn, ldn, i, p, (x[i] * r) * w[i]);
    }
}

// One add-norm launch of a pass of P columns (the variant and the PDL flag of
// the pass: programmatic chaining pays in a batched decode step, and costs a
// prefill chunk's multi-wave grids more than it saves).
int add_norm(int P, bool pdl, cudaStream_t st, float* X, const float* Yp, int parts, size_t split_stride,
             const float* w, float* Xn, int ldn, int H, float eps, const HOut& ho) {
    if (P <= kMaxSeg && H <= 4 * kAddNormWide)  // up to 4 values per thread: the parts' loads stay in registers
        return launch_pdl(pf_add_norm_kernel<true, 4>, dim3(P), dim3(kAddNormWide), 0, st, pdl, X, Yp, parts,
                          split_stride, w, Xn, ldn, H, eps, ho);
    if (P <= kMaxSeg)
        return launch_pdl(pf_add_norm_kernel<true, kAddNormPer>, dim3(P), dim3(kAddNormWide), 0, st, pdl, X, Yp, parts,
                          split_stride, w, Xn, ldn, H, eps, ho);
    return launch_pdl(pf_add_norm_kernel<false>, dim3(P), dim3(256), 0, st, pdl, X, Yp, parts, split_stride, w, Xn, ldn,
                      H, eps, ho);
}

// Causal conv1d + SiLU of the qkv rows and the alpha/beta gates, one thread
// per (token, row): the conv of token p reads inputs p-K+1..p (older ones from
// the window of the previous call), taps in the decode step's order; no
// recurrence, so the whole chunk runs at once.  Z rows [qkv C | alpha nv |
// beta nv | z].  The window moves afterwards (pf_conv_window_kernel).
__global__ void pf_conv_gates_kernel(const float* Z, int ldz, int P, int C, int nv, int K,
                                     const Segs sg, const float* wconv,
                                     const float* dt_bias, const float* a,
                                     float* Cq, float* dt, float* beta) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int W = C + nv;
    if (idx >= static_cast<long long>(P) * W) return;
    const int p = static_cast<int>(idx / W), c = static_cast<int>(idx - static_cast<long long>(p) * W);
    if (c < C) {
        const int s = seg_of(sg, p), c0 = sg.col0[s];  // inputs before the segment's first column: its window
        const float* win = sg.conv[s];
        const float* kw = wconv + static_cast<size_t>(c) * K;
        float acc = 0.0f;
        for (int t = 0; t < K - 1; ++t) {
            const int i = p - (K - 1) + t;
            const float x = i >= c0 ? Z[static_cast<size_t>(i) * ldz + c]
                                    : win[static_cast<size_t>(c) * (K - 1) + (K - 1) + (i - c0)];
            acc += kw[t] * x;
        }
        acc += kw[K - 1] * Z[static_cast<size_t>(p) * ldz + c];
        Cq[static_cast<size_t>(p) * C + c] = silu(acc);
    } else {
        const int h = c - C;  // dt = softplus(alpha + dt_bias) * a, beta = sigmoid(beta_raw)
        dt[p * nv + h] = softplus(Z[static_cast<size_t>(p) * ldz + C + h] + dt_bias[h]) * a[h];
        beta[p * nv + h] = sigmoid(Z[static_cast<size_t>(p) * ldz + C + nv + h]);
    }
}

// The same for a pass of one sequence (one segment starting at column 0)
// with K = 4 taps: thread (channel c, block of kConvTB columns) keeps the
// channel's taps and the block's inputs (and the 3 before it) in registers,
// so each input is read once per block instead of once per tap; the gate
// columns c >= C give dt and beta of the block's columns.  Same sums in the
// same order as pf_conv_gates_kernel.  Grid (ceil((C + nv) / 256), ceil(P / kConvTB)).
constexpr int kConvTB = 16;
__global__ void pf_conv4_block_kernel(const float* Z, int ldz, int P, int C, int nv, const float* win,
                                      const float* wconv, const float* dt_bias, const float* a, float* Cq,
                                      float* dt, float* beta) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    const int c = blockIdx.x * blockDim.x + threadIdx.x, p0 = blockIdx.y * kConvTB;
    if (c >= C + nv) return;
    if (c >= C) {
        const int h = c - C;  // dt = softplus(alpha + dt_bias) * a, beta = sigmoid(beta_raw)
        for (int p = p0; p < min(P, p0 + kConvTB); ++p) {
            dt[p * nv + h] = softplus(Z[static_cast<size_t>(p) * ldz + C + h] + dt_bias[h]) * a[h];
            beta[p * nv + h] = sigmoid(Z[static_cast<size_t>(p) * ldz + C + nv + h]);
        }
        return;
    }
    float w[4], x[kConvTB + 3];
#pragma unroll
    for (int t = 0; t < 4; ++t) w[t] = wconv[static_cast<size_t>(c) * 4 + t];
#pragma unroll
    for (int i = 0; i < 3; ++i) {  // the inputs before the block (the window before column 0)
        const int q = p0 - 3 + i;
        x[i] = q >= 0 ? Z[static_cast<size_t>(q) * ldz + c] : win[static_cast<size_t>(c) * 3 + 3 + q];
    }
#pragma unroll
    for (int i = 0; i < kConvTB; ++i) {
        const int q = p0 + i;
        x[3 + i] = q < P ? Z[static_cast<size_t>(q) * ldz + c] : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < kConvTB; ++i) {
        if (p0 + i >= P) break;
        float acc = 0.0f;
#pragma unroll
        for (int t = 0; t < 3; ++t) acc += w[t] * x[i + t];
        acc += w[3] * x[i + 3];
        Cq[static_cast<size_t>(p0 + i) * C + c] = silu(acc);
    }
}

// Each segment's conv window after the pass: its last K-1 inputs, oldest
// first (from the old window where the segment is shorter than that).  Grid
// (rows / 256, segments).
__global__ void pf_conv_window_kernel(const float* Z, int ldz, int C, int K, const Segs sg) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    const int c = blockIdx.x * blockDim.x + threadIdx.x, s = blockIdx.y;
    if (c >= C) return;
    const int c0 = sg.col0[s], P = sg.col0[s + 1] - c0;
    float nw[kMaxConvTaps];
    float* wc = sg.conv[s] + static_cast<size_t>(c) * (K - 1);
    for (int t = 0; t < K - 1; ++t) {
        const int i = P - (K - 1) + t;
        nw[t] = i >= 0 ? Z[static_cast<size_t>(c0 + i) * ldz + c] : wc[(K - 1) + i];
    }
    for (int t = 0; t < K - 1; ++t) wc[t] = nw[t];
}

// Per-head L2 norm of each token's q and k (head_k_dim 128): one warp per
// (token, q|k, key head); QKn [P][2][nk][128].
__global__ void pf_l2norm_kernel(const float* Cq, int C, int kdim, int nk, int P, float eps,
                                 float* QKn) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (wid >= P * 2 * nk) return;
    const int p = wid / (2 * nk), r = wid - p * 2 * nk, which = r / nk, kh = r - which * nk;
    const float4 v = *reinterpret_cast<const float4*>(Cq + static_cast<size_t>(p) * C + which * kdim + kh * kDk + 4 * lane);
    float ss = v.x * v.x;
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
    ss = warp_sum(ss);
    const float rr = 1.0f / sqrtf(ss + eps);
    *reinterpret_cast<float4*>(QKn + (static_cast<size_t>(wid)) * kDk + 4 * lane) =
        make_float4(v.x * rr, v.y * rr, v.z * rr, v.w * rr);
}

// The delta rule over the chunk: CTA = 32 state rows of one value head, each
// warp 4 rows held in registers (lane: dims 4 lane..+3) for the whole chunk;
// per token decay, read, rank-1 update and query as the decode step does
// (delta_rows4), with the decay applied to the read's sum (g (S k)) and each
// token's query reduced together with the next token's read, so that only
// the read's reduction lies on the state's chain from token to token.  The
// inputs of 16 tokens at a time (the head's normalised q and k, the CTA's v
// values, the decay factors and gates) are staged in shared memory by the
// whole CTA, two stages deep (the next stage's async copies run under this
// stage's tokens), so the token loop reads shared memory only.  O [P][v_dim].
constexpr int kDeltaStage = 16;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__global__ void __launch_bounds__(256) pf_delta_kernel(const float* Cq_all, int C, int kdim,
                                                       const float* QKn_all,
                                                       const float* dt_all,
                                                       const float* beta_all, const Segs sgs,
                                                       float* O_all, int nk, int nv, int dv) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    // segment blockIdx.y: its columns c0.. and its recurrent state
    const int c0 = sgs.col0[blockIdx.y], P = sgs.col0[blockIdx.y + 1] - c0;
    float* S = sgs.ssm[blockIdx.y];
    const float* Cq = Cq_all + static_cast<size_t>(c0) * C;
    const float* QKn = QKn_all + static_cast<size_t>(c0) * 2 * nk * kDk;
    const float* dt = dt_all + c0 * nv;
    const float* beta = beta_all + c0 * nv;
    float* O = O_all + static_cast<size_t>(c0) * nv * dv;
    // two stages: the next one's inputs arrive while this one's tokens run
    __shared__ __align__(16) float sq[2][kDeltaStage][kDk];
    __shared__ __align__(16) float sk[2][kDeltaStage][kDk];
    __shared__ __align__(16) float sv[2][kDeltaStage][32];  // rows read as float4 by each warp
    __shared__ float sg[2][kDeltaStage], sb[2][kDeltaStage];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per_head = dv / 32;
    const int h = blockIdx.x / per_head, jb = (blockIdx.x - h * per_head) * 32, j = jb + 4 * warp;
    const int kh = h % nk;
    const int vd = nv * dv;
    // async copies of tokens p1 .. p1 + kDeltaStage - 1 (those before P) into stage buffer b:
    // the head's normalised q and k rows and the CTA's 32 v values (16-byte pieces)
    auto issue_stage = [&](int p1, int b) {
        const int n1 = min(kDeltaStage, P - p1);
        for (int e = tid; e < n1 * 64; e += 256) {
            const int t = e >> 6, r = e & 63, which = r >> 5, c4 = r & 31;
            cp_async16((which ? &sk[b][t][0] : &sq[b][t][0]) + 4 * c4,
                       QKn + (static_cast<size_t>(p1 + t) * 2 * nk + which * nk + kh) * kDk + 4 * c4);
        }
        for (int e = tid; e < n1 * 8; e += 256) {
            const int t = e >> 3, c4 = e & 7;
            cp_async16(&sv[b][t][4 * c4], Cq + static_cast<size_t>(p1 + t) * C + 2 * kdim + h * dv + jb + 4 * c4);
        }
    };
    issue_stage(0, 0);
    if (tid < min(kDeltaStage, P)) {
        sg[0][tid] = expf(dt[tid * nv + h]);  // the decay factor, off the token loop's chain
        sb[0][tid] = beta[tid * nv + h];
    }
    float4 st[4];
    float* Sg = S + (static_cast<size_t>(h) * dv + j) * kDk;
#pragma unroll
    for (int t = 0; t < 4; ++t) st[t] = *reinterpret_cast<const float4*>(Sg + t * kDk + 4 * lane);
    const float scale = 1.0f / sqrtf(static_cast<float>(kDk));
    float oq[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // the pending token's query partial sums
    int pend = -1;                          // its column, -1: none
    cp_async_wait_all();
    __syncthreads();
    for (int p0 = 0, cur = 0; p0 < P; p0 += kDeltaStage, cur ^= 1) {
        const int np = min(kDeltaStage, P - p0), p1 = p0 + kDeltaStage;
        // the next stage: its copies in flight, its gates in registers (the
        // exponential taken after this stage's tokens, off their chain)
        float gn = 0.0f, bn = 0.0f;
        const bool more = p1 < P;
        if (more) {
            issue_stage(p1, cur ^ 1);
            if (tid < min(kDeltaStage, P - p1)) {
                gn = dt[(p1 + tid) * nv + h];
                bn = beta[(p1 + tid) * nv + h];
            }
        }
        const float(*sq_c)[kDk] = sq[cur];
        const float(*sk_c)[kDk] = sk[cur];
        const float(*sv_c)[32] = sv[cur];
        const float* sg_c = sg[cur];
        const float* sb_c = sb[cur];
        for (int t = 0; t < np; ++t) {
            const float4 kk = *reinterpret_cast<const float4*>(&sk_c[t][4 * lane]);
            const float4 qq = *reinterpret_cast<const float4*>(&sq_c[t][4 * lane]);
            const float4 vv = *reinterpret_cast<const float4*>(&sv_c[t][4 * warp]);  // the warp's 4 v values
            const float gd = sg_c[t], be = sb_c[t];
            float a[8];  // the read's partial sums (this token), the query's (the pending token)
#pragma unroll
            for (int u = 0; u < 4; ++u) {  // read: (g S) k = g (S k), the decay applied to the sum
                float d = st[u].x * kk.x;
                d = fmaf(st[u].y, kk.y, d);
                d = fmaf(st[u].z, kk.z, d);
                a[u] = fmaf(st[u].w, kk.w, d);
                a[4 + u] = oq[u];
            }
            // the eight sums over the warp in one transposed xor tree (lanes
            // paired 16, 8, 4, 2, 1 apart as in a plain tree, the same sums):
            // each level a lane keeps half of its values and adds the
            // partner's copy of them; at the end lane l holds sum number
            // 4 (l >> 4 & 1) + 2 (l >> 3 & 1) + (l >> 2 & 1)
            const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
            float r4[4], r2[2];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                r4[i] = (b4 ? a[4 + i] : a[i]) + __shfl_xor_sync(0xffffffffu, b4 ? a[i] : a[4 + i], 16);
#pragma unroll
            for (int i = 0; i < 2; ++i)
                r2[i] = (b3 ? r4[2 + i] : r4[i]) + __shfl_xor_sync(0xffffffffu, b3 ? r4[i] : r4[2 + i], 8);
            float r1 = (b2 ? r2[1] : r2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? r2[0] : r2[1], 4);
            r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
            r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
            // read sum u sits in lane 8 (u >> 1) + 4 (u & 1), query sum u 16 lanes on
            if (pend >= 0 && b4 && (lane & 3) == 0)
                O[static_cast<size_t>(pend) * vd + h * dv + j + ((lane >> 2) & 3)] = r1 * scale;
            float dot[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) dot[u] = __shfl_sync(0xffffffffu, r1, 8 * (u >> 1) + 4 * (u & 1));
            const float vl[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float d = be * (vl[u] - gd * dot[u]);
                st[u] = make_float4(fmaf(kk.x, d, gd * st[u].x), fmaf(kk.y, d, gd * st[u].y),
                                    fmaf(kk.z, d, gd * st[u].z), fmaf(kk.w, d, gd * st[u].w));  // decay + rank-1 update
                float q = st[u].x * qq.x;
                q = fmaf(st[u].y, qq.y, q);
                q = fmaf(st[u].z, qq.z, q);
                oq[u] = fmaf(st[u].w, qq.w, q);  // query, reduced with the next token's read
            }
            pend = p0 + t;
        }
        if (more && tid < min(kDeltaStage, P - p1)) {
            sg[cur ^ 1][tid] = expf(gn);
            sb[cur ^ 1][tid] = bn;
        }
        cp_async_wait_all();
        __syncthreads();  // the next stage is in; this one is no longer read (its buffer is refilled next)
    }
    if (pend >= 0) {  // the last token's query
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int u = 0; u < 4; ++u) oq[u] += __shfl_xor_sync(0xffffffffu, oq[u], off);
        float mine = 0.0f;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (lane == u) mine = oq[u] * scale;
        if (lane < 4) O[static_cast<size_t>(pend) * vd + h * dv + j + lane] = mine;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) *reinterpret_cast<float4*>(Sg + u * kDk + 4 * lane) = st[u];
}

// Gated RMSNorm per value head: U = RMSNorm(o_h) * w * silu(z_h), into column
// p of the GEMM input U (put_in).  Grid (P, ceil(nv / 8)), one warp per head
// (head_v_dim 32/64/128: 1, 2 or 4 values per lane).
__global__ void __launch_bounds__(256) pf_gated_norm_kernel(const float* O, const float* Z,
                                                            int ldz, int zoff, const float* w, int nv,
                                                            int dv, float eps, float* U, int ldu) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    const int p = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per = dv / 32;
    const int h = 8 * blockIdx.y + warp;
    if (h >= nv) return;
    const float* o = O + static_cast<size_t>(p) * nv * dv + h * dv;
    const float* z = Z + static_cast<size_t>(p) * ldz + zoff + h * dv;
    float ov[4], ss = 0.0f;
    for (int e = 0; e < per; ++e) {
        ov[e] = o[lane + 32 * e];
        ss = fmaf(ov[e], ov[e], ss);
    }
    ss = warp_sum(ss);
    const float rn = 1.0f / sqrtf(ss / static_cast<float>(dv) + eps);
    for (int e = 0; e < per; ++e) {
        const int i = lane + 32 * e;
        put_in(U, ldu, h * dv + i, p, ((ov[e] * rn) * w[i]) * silu(z[i]));
    }
}

// Attention inputs of token p (position pos0 + p): per-head RMSNorm and
// partial NEOX rope of q (to Qn [P][nh][256]) and k, and the K and V rows
// (to the f32 cache rows, or to staging rows for the quantizer).  Grid P.
__global__ void __launch_bounds__(256) pf_attn_prep_kernel(const float* Z, int ldz, int nh, int nkv,
                                                           const float* q_norm,
                                                           const float* k_norm, const Segs sg, int n_rot,
                                                           float theta_scale, float eps, float* Qn,
                                                           float* Kst, float* Vst) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    __shared__ float cs[kHd / 2], sn[kHd / 2];
    __shared__ __align__(16) float vec[8][kHd];
    const int p = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = n_rot / 2, qd = nh * kHd, kvd = nkv * kHd;
    const int s = seg_of(sg, p);
    const int pos = sg.pos0[s] + (p - sg.col0[s]);
    // K/V rows: straight into the sequence's f32 cache row pos, or (staging
    // given) into column p of the staging rows for the quantizer
    float* Krow = Kst ? Kst + static_cast<size_t>(p) * kvd : sg.kc[s] + static_cast<size_t>(pos) * kvd;
    float* Vrow = Vst ? Vst + static_cast<size_t>(p) * kvd : sg.vc[s] + static_cast<size_t>(pos) * kvd;
    if (tid < half) {  // theta_0 = pos, theta_{i+1} = theta_i * theta_scale (f32 running product)
        float th = static_cast<float>(pos);
        for (int i = 0; i < tid; ++i) th = th * theta_scale;
        float sv, cv;
        sincosf(th, &sv, &cv);
        cs[tid] = cv;
        sn[tid] = sv;
    }
    const float* z = Z + static_cast<size_t>(p) * ldz;
    for (int i = tid; i < kvd; i += 256) Vrow[i] = z[2 * qd + kvd + i];
    __syncthreads();
    for (int job0 = 0; job0 < nh + nkv; job0 += 8) {
        const int job = job0 + warp;
        if (job < nh + nkv) {
            const float* src = job < nh ? z + static_cast<size_t>(job) * 2 * kHd : z + 2 * qd + (job - nh) * kHd;
            const float* w = job < nh ? q_norm : k_norm;
            float v[8];
            row8(src, lane, v);
            float ss = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
            ss = warp_sum(ss);
            const float r = 1.0f / sqrtf(ss / static_cast<float>(kHd) + eps);
#pragma unroll
            for (int i = 0; i < 8; ++i) vec[warp][dim8(lane, i)] = (v[i] * r) * w[dim8(lane, i)];
            __syncwarp();
            for (int i = lane; i < half; i += 32) {
                const float x0 = vec[warp][i], x1 = vec[warp][i + half];
                vec[warp][i] = x0 * cs[i] - x1 * sn[i];
                vec[warp][i + half] = x0 * sn[i] + x1 * cs[i];
            }
            __syncwarp();
            float* dst = job < nh ? Qn + (static_cast<size_t>(p) * nh + job) * kHd : Krow + (job - nh) * kHd;
            for (int i = lane; i < kHd; i += 32) dst[i] = vec[warp][i];
            __syncwarp();
        }
    }
}

// Causal GQA attention of the chunk's tokens: CTA (p, g, z) for the GS query
// heads of kv group g of token p over cache rows 0..pos0+p (f32 rows, or
// quantized records read dequantized), 8 warps taking keys t = warp mod 8 with
// an online softmax each, then combined.  Without Part (grid z = 1): the
// output is gated by sigmoid(gate) and stored to column p of the GEMM input
// Att (put_in).  With Part (a batched decode step, grid z = the key
// splits): CTA z takes the z-th of gridDim.z equal runs of the rows and stores
// its running max, sum and unnormalised output per head to Part (merged by
// pf_attn_merge_kernel).
template <int GS, bool KVQ>
__global__ void __launch_bounds__(256) pf_causal_attn_kernel(const float* Qn, const float* Z,
                                                             int ldz, const Segs sg, int kvd,
                                                             float* Att, int lda,
                                                             float* Part) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    __shared__ float wml[8][GS][2];
    __shared__ __align__(16) float wacc[8][GS][kHd];
    const int p = blockIdx.x, g = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sq = seg_of(sg, p);
    const float* kc = sg.kc[sq];
    const float* vc = sg.vc[sq];
    const int max_seq = sg.max_seq[sq];
    const int nh = gridDim.y * GS, t_len = sg.pos0[sq] + (p - sg.col0[sq]) + 1;
    float q[GS][8], m[GS], l[GS], acc[GS][8];
#pragma unroll
    for (int i = 0; i < GS; ++i) {
        row8(Qn + (static_cast<size_t>(p) * nh + g * GS + i) * kHd, lane, q[i]);
        m[i] = -INFINITY;
        l[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
    }
    const float scale = 1.0f / sqrtf(static_cast<float>(kHd));
    const int per = (t_len + gridDim.z - 1) / gridDim.z, t_lo = blockIdx.z * per, t_hi = min(t_len, t_lo + per);
    for (int t = t_lo + warp; t < t_hi; t += 8) {
        float kv[8], vv[8];
        if constexpr (KVQ) {
            const size_t rec = static_cast<size_t>(g) * max_seq + t;
            kvq_k8(reinterpret_cast<const uint8_t*>(kc) + rec * kKRec, lane, kv);
            kvq_v8(reinterpret_cast<const uint8_t*>(vc) + rec * kVRec, lane, vv);
        } else {
            load_row8(kc + static_cast<size_t>(t) * kvd + g * kHd, lane, kv);
            load_row8(vc + static_cast<size_t>(t) * kvd + g * kHd, lane, vv);
        }
#pragma unroll
        for (int i = 0; i < GS; ++i) {
            float dot = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) dot = fmaf(q[i][j], kv[j], dot);
            const float sc = warp_sum(dot) * scale;
            const float mn = fmaxf(m[i], sc);
            const float c = expf(m[i] - mn), pr = expf(sc - mn);
            l[i] = fmaf(l[i], c, pr);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(acc[i][j], c, pr * vv[j]);
            m[i] = mn;
        }
    }
#pragma unroll
    for (int i = 0; i < GS; ++i) {
        if (lane == 0) {
            wml[warp][i][0] = m[i];
            wml[warp][i][1] = l[i];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) wacc[warp][i][dim8(lane, j)] = acc[i][j];
    }
    __syncthreads();
    for (int i = 0; i < GS; ++i) {  // thread tid owns dim tid of every head
        float M = -INFINITY;
        for (int w = 0; w < 8; ++w) M = fmaxf(M, wml[w][i][0]);
        float L = 0.0f, A = 0.0f;
        for (int w = 0; w < 8; ++w) {
            const float mw = wml[w][i][0];
            const float f = mw == -INFINITY ? 0.0f : expf(mw - M);
            L = fmaf(wml[w][i][1], f, L);
            A = fmaf(wacc[w][i][tid], f, A);
        }
        const int h = g * GS + i;
        if (Part) {  // [p][h][z]: kHd outputs, then max and sum
            float* pr = Part + ((static_cast<size_t>(p) * nh + h) * gridDim.z + blockIdx.z) * (kHd + 2);
            pr[tid] = A;
            if (tid == 0) {
                pr[kHd] = M;
                pr[kHd + 1] = L;
            }
        } else {
            const float gt = Z[static_cast<size_t>(p) * ldz + static_cast<size_t>(h) * 2 * kHd + kHd + tid];
            put_in(Att, lda, h * kHd + tid, p, (A / L) * sigmoid(gt));
        }
    }
}

// The key splits of pf_causal_attn_kernel's Part merged (split order) and
// gated: CTA (p, h), thread tid = output dim.  An empty split has max -inf.
__global__ void __launch_bounds__(kHd) pf_attn_merge_kernel(const float* Part, int splits,
                                                            const float* Z, int ldz,
                                                            float* Att, int lda) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    const int p = blockIdx.x, h = blockIdx.y, nh = gridDim.y, tid = threadIdx.x;
    const float* pr = Part + (static_cast<size_t>(p) * nh + h) * splits * (kHd + 2);
    // every split's loads in flight at once (splits <= kAttnSplits), then the
    // merge in split order
    float ms[kAttnSplits], ls[kAttnSplits], as[kAttnSplits];
#pragma unroll
    for (int z = 0; z < kAttnSplits; ++z) {
        const bool in = z < splits;
        ms[z] = in ? pr[z * (kHd + 2) + kHd] : -INFINITY;
        ls[z] = in ? pr[z * (kHd + 2) + kHd + 1] : 0.0f;
        as[z] = in ? pr[z * (kHd + 2) + tid] : 0.0f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int z = 0; z < kAttnSplits; ++z) M = fmaxf(M, ms[z]);
    float L = 0.0f, A = 0.0f;
#pragma unroll
    for (int z = 0; z < kAttnSplits; ++z) {
        if (z >= splits) break;
        const float f = ms[z] == -INFINITY ? 0.0f : expf(ms[z] - M);
        L = fmaf(ls[z], f, L);
        A = fmaf(as[z], f, A);
    }
    const float gt = Z[static_cast<size_t>(p) * ldz + static_cast<size_t>(h) * 2 * kHd + kHd + tid];
    put_in(Att, lda, h * kHd + tid, p, (A / L) * sigmoid(gt));
}

// A = silu(G) * U, elementwise over P columns of ffn values, G and U given as
// split sums (added in order): ldk > 0, k-major [ffn][ldk] (a batched decode
// step, thread e on value e / P of column e % P); ldk == 0, token-major [P][ffn]
// (a prefill chunk: consecutive threads on consecutive values of one token, so
// the tile stores of put_xt stay within 128-byte rows).  A is a GEMM input
// (put_in: k-major [ffn][lda], or lda == 0 the tensor-core tiles).
__global__ void pf_swiglu_kernel(const float* Gp, int gparts, const float* Up, int uparts,
                                 size_t stride, float* A, int ffn, int P, int ldk, int lda) {
    pdl_launch_dependents();  // the next kernel of the pass may start its prologue
    pdl_wait();               // everything earlier in the pass is complete and visible
    const size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= static_cast<size_t>(ffn) * P) return;
    const int kk = ldk ? static_cast<int>(e / P) : static_cast<int>(e % ffn);
    const int p = ldk ? static_cast<int>(e % P) : static_cast<int>(e / ffn);
    const size_t i = ldk ? static_cast<size_t>(kk) * ldk + p : static_cast<size_t>(p) * ffn + kk;
    float g = Gp[i], u = Up[i];
    const int parts = max(gparts, uparts);
    for (int z0 = 1; z0 < parts; z0 += 4) {  // both sums' loads in flight, each added in part order
        float tg[4], tu[4];
#pragma unroll
        for (int zz = 0; zz < 4; ++zz) {
            tg[zz] = z0 + zz < gparts ? Gp[(z0 + zz) * stride + i] : 0.0f;
            tu[zz] = z0 + zz < uparts ? Up[(z0 + zz) * stride + i] : 0.0f;
        }
#pragma unroll
        for (int zz = 0; zz < 4; ++zz) {
            if (z0 + zz < gparts) g += tg[zz];
            if (z0 + zz < uparts) u += tu[zz];
        }
    }
    put_in(A, lda, kk, p, silu(g) * u);
}

// ------------------------------------------------------------ host side
struct Scratch {
    int chunk;
    int* tok;
    // Xn, Uin and A are GEMM inputs: f32 [k][4] for a batched decode step, the
    // put_xt tiles (kXtBytesPerValue bytes a value) for a prefill chunk
    float *X, *Xn, *Z, *Yp, *Zp, *Up, *A, *Cq, *dt, *beta, *QKn, *O, *Uin, *Qn, *Ks, *Vs;
    float* Ap;  // the attention's key-split partials of a batched decode step [kSmallBatch][n_heads][kAttnSplits][kHd + 2]
    size_t cap_yp, cap_zp, cap_up;  // floats of the split-sum buffers Yp, Zp, Up
    int* pos;  // device: the pass's first position per segment [kMaxSeg]
};

template <class T>
int pf_alloc(qg_state* s, T** p, size_t count) {
    void* q = nullptr;
    cudaError_t e = cudaMalloc(&q, (count ? count : 1) * sizeof(T));
    if (e != cudaSuccess) return set_err(QG_ERR_OOM, "prefill: cudaMalloc of %zu bytes: %s", count * sizeof(T),
                                         cudaGetErrorString(e));
    s->allocs.push_back(q);
    s->stats.device_allocs++;
    *p = static_cast<T*>(q);
    return QG_OK;
}

size_t split_rows(int n, int k, int P);

int scratch_of(const qg_model* m, qg_state* s, Scratch** out) {
    if (s->pf) {
        *out = static_cast<Scratch*>(s->pf);
        return QG_OK;
    }
    const qg_config& c = m->cfg;
    const size_t P = kPfChunk, H = c.hidden;
    size_t n_in = 0;
    for (int il = 0; il < c.n_layers; ++il) n_in = std::max(n_in, static_cast<size_t>(m->layers[il].n_in));
    const size_t mid = std::max({static_cast<size_t>(m->v_dim), static_cast<size_t>(m->q_dim), size_t(1)});
    // the split-sum buffers: as many [n] vectors as the largest split layout
    // any projection of the model takes for any pass of 1..kPfChunk columns
    // (the rule of splits_for; gemm refuses a layout past these sizes)
    // (per buffer: Yp takes the output projections and ffn_down, Zp the input
    // projections and the gate, Up the up projection)
    size_t rows_y = 1, rows_z = 1, rows_u = 1;
    for (int il = 0; il < c.n_layers; ++il) {
        const qg_layer_dev& L = m->layers[il];
        const int k_out = m->kinds[il] == QG_LAYER_DELTANET ? m->v_dim : m->q_dim;
        for (int p = 1; p <= kPfChunk; ++p) {
            rows_y = std::max({rows_y, split_rows(c.hidden, k_out, p), split_rows(c.hidden, c.ffn, p)});
            rows_z = std::max({rows_z, split_rows(L.n_in, c.hidden, p), split_rows(c.ffn, c.hidden, p)});
            rows_u = std::max(rows_u, split_rows(c.ffn, c.hidden, p));
        }
    }
    Scratch* sc = new (std::nothrow) Scratch();
    if (!sc) return set_err(QG_ERR_OOM, "prefill: host allocation");
    sc->chunk = kPfChunk;
    sc->cap_yp = rows_y * H;
    sc->cap_zp = rows_z * std::max(n_in, static_cast<size_t>(c.ffn));
    sc->cap_up = rows_u * c.ffn;
    int rc = QG_OK;
    (void)((rc = pf_alloc(s, &sc->tok, P)) || (rc = pf_alloc(s, &sc->pos, kMaxSeg)) || (rc = pf_alloc(s, &sc->X, P * H)) || (rc = pf_alloc(s, &sc->Xn, P * H * kXtBytesPerValue / 4)) ||
           (rc = pf_alloc(s, &sc->Z, P * n_in)) || (rc = pf_alloc(s, &sc->Yp, sc->cap_yp)) ||
           (rc = pf_alloc(s, &sc->Zp, sc->cap_zp)) || (rc = pf_alloc(s, &sc->Up, sc->cap_up)) ||
           (rc = pf_alloc(s, &sc->A, P * c.ffn * kXtBytesPerValue / 4)) || (rc = pf_alloc(s, &sc->Cq, P * std::max(m->conv_dim, 1))) ||
           (rc = pf_alloc(s, &sc->dt, P * (c.n_v_heads + 1))) || (rc = pf_alloc(s, &sc->beta, P * (c.n_v_heads + 1))) ||
           (rc = pf_alloc(s, &sc->QKn, P * 2 * std::max(m->k_dim, 1))) ||
           (rc = pf_alloc(s, &sc->O, P * std::max(m->v_dim, 1))) || (rc = pf_alloc(s, &sc->Uin, P * mid * kXtBytesPerValue / 4)) ||
           (rc = pf_alloc(s, &sc->Qn, P * std::max(m->q_dim, 1))) || (rc = pf_alloc(s, &sc->Ks, P * std::max(m->kv_dim, 1))) ||
           (rc = pf_alloc(s, &sc->Vs, P * std::max(m->kv_dim, 1))) ||
           (rc = pf_alloc(s, &sc->Ap, static_cast<size_t>(kSmallBatch) * std::max(c.n_heads, 1) * kAttnSplits * (kHd + 2))));
    if (rc) {
        delete sc;
        return rc;
    }
    s->pf = sc;
    *out = sc;
    return QG_OK;
}

// An upper bound on the K slices of the small-batch GEMV over k inputs (one
// output part each): slices of 2048, then at most three for the remainder's
// binary digits (1024, 512, 256).
inline int max_slices(int k) { return k / 2048 + 3; }

// Y = W X: for at most kSmallBatch columns (a batched decode step) X packed
// k-major [k][4] (P <= 4) or [k][8], and the small-batch GEMV once per group of
// 4 columns; else X as the tensor-core tiles of put_xt and pf_mma_kernel.
// ROW_MAJOR: Y[row][ldy] per split (split stride n * ldy), else Y[token][ldy]
// (split stride P * ldy).
template <int QT, bool ROW_MAJOR>
int gemm(const uint8_t* W, int n, int k, const float* X, float* Y, int ldy, int P, int splits, cudaStream_t st,
         int* used_splits, unsigned* err, size_t cap) {
    if (P <= kSmallBatch) {  // a batched decode step: the small-batch GEMV per 4 columns, one part per K slice
        const size_t split_stride = ROW_MAJOR ? static_cast<size_t>(n) * ldy : static_cast<size_t>(P) * ldy;
        if (static_cast<size_t>(max_slices(k)) * split_stride > cap)
            return set_err(QG_ERR_SHAPE, "prefill: the slice sums of a %d x %d GEMV exceed their buffer", n, k);
        const int xq = P <= 4 ? 4 : 8;
        int parts = 1;
        for (int g = 0; 4 * g < P; ++g) {
            float* Yg = ROW_MAJOR ? Y + 4 * g : Y + static_cast<size_t>(4 * g) * ldy;
            if (int rc = launch_bm4<QT, ROW_MAJOR, false>(W, n, k, X + 4 * g, xq, Yg, ldy, split_stride,
                                                          std::min(4, P - 4 * g), BmArgmax{}, err, st, &parts))
                return rc;
        }
        if (used_splits) *used_splits = parts;
        return QG_OK;
    }
    const int nq = k / 64;
    if (splits > nq) splits = nq;
    if (splits < 1) splits = 1;
    const int per = (nq + splits - 1) / splits;
    const int z = (nq + per - 1) / per;
    if (used_splits) *used_splits = z;
    const size_t split_stride = ROW_MAJOR ? static_cast<size_t>(n) * ldy : static_cast<size_t>(P) * ldy;
    if (static_cast<size_t>(z) * split_stride > cap)
        return set_err(QG_ERR_SHAPE, "prefill: %d K splits of a %d x %d GEMM exceed their buffer", z, n, k);
    if (int rc = grant_smem(reinterpret_cast<const void*>(pf_mma_kernel<QT, ROW_MAJOR>), kMmaSmem)) return rc;
    const dim3 grid((n + 127) / 128, (P + 255) / 256, z);
    if (int e_ = launch_pdl(pf_mma_kernel<QT, ROW_MAJOR>, grid, dim3(kMmaThreads), kMmaSmem, st, false, W, n, k,
                            reinterpret_cast<const uint8_t*>(X), Y, ldy, split_stride, P, per, err))
        return e_;
    return QG_OK;
}

// K splits of a projection (one CTA per SM at a time).  Fewer row x 256-token
// tiles than SMs: the split count, up to kPfMaxSplit with at least 8
// quarters (512 inputs) a split, whose CTAs best fill their waves of SMs, a
// further split only where it fills 10 points more.  Otherwise a second split
// only where it cuts the SMs left idle by the last wave by 10 points or more
// and K holds 32 quarters: the CTA's fixed costs (tensor memory, pipeline
// fill, the output tile) stay small against its K loop.
int splits_for(int n, int k, int P) {
    const long long ctas = static_cast<long long>((n + 127) / 128) * ((P + 255) / 256), sms = device_sms();
    auto eff = [&](long long z) {
        const long long c = ctas * z, waves = (c + sms - 1) / sms;
        return static_cast<double>(c) / static_cast<double>(waves * sms);
    };
    if (ctas < sms) {
        const int zmax = std::max(1, std::min(kPfMaxSplit, k / 64 / 8));
        int best = 1;
        for (int z = 2; z <= zmax; ++z)
            if (eff(z) > eff(best) + 0.1) best = z;
        return best;
    }
    return (k / 64 >= 32 && eff(2) > eff(1) + 0.1) ? 2 : 1;
}

// Columns' worth of split partial sums a projection n x k writes for a pass of
// P columns (the split buffers hold this many [n] vectors): one part per K
// slice of [n][8] (row-major) or [P][n] for a batched decode step, else the K
// splits gemm takes of [P][n] each.
size_t split_rows(int n, int k, int P) {
    if (P <= kSmallBatch) return static_cast<size_t>(max_slices(k)) * kSmallBatch;
    const int nq = k / 64;
    const int splits = std::min(std::max(splits_for(n, k, P), 1), nq);
    const int per = (nq + splits - 1) / splits;
    return static_cast<size_t>((nq + per - 1) / per) * P;
}

template <bool KVQ>
int launch_causal(int gs, dim3 grid, cudaStream_t st, bool pdl, const float* Qn, const float* Z, int ldz, const Segs& sg,
                  int kvd, float* att, int ldk, float* part) {
    switch (gs) {
        case 1:
            return launch_pdl(pf_causal_attn_kernel<1, KVQ>, grid, dim3(256), 0, st, pdl, Qn, Z, ldz, sg, kvd, att, ldk,
                              part);
        case 2:
            return launch_pdl(pf_causal_attn_kernel<2, KVQ>, grid, dim3(256), 0, st, pdl, Qn, Z, ldz, sg, kvd, att, ldk,
                              part);
        case 4:
            return launch_pdl(pf_causal_attn_kernel<4, KVQ>, grid, dim3(256), 0, st, pdl, Qn, Z, ldz, sg, kvd, att, ldk,
                              part);
        default: return set_err(QG_ERR_SHAPE, "prefill: GQA group of %d query heads is not served", gs);
    }
}

// One pass of columns through every layer: segment i is sequence ss[i]'s
// tokens at positions pos0[i].. in columns col0[i]..col0[i+1]-1 (token ids in
// sc->tok).  X holds each column's residual stream at the end.
struct Pass {
    int n;
    qg_state* ss[kMaxSeg];
    const int* pos_dev;  // device: first position of each segment
    int col0[kMaxSeg + 1];
};

Segs segs_of(const Pass& ps, int il) {
    Segs sg{};
    sg.n = ps.n;
    for (int i = 0; i < ps.n; ++i) {
        sg.col0[i] = ps.col0[i];
        sg.max_seq[i] = ps.ss[i]->max_seq;
        sg.conv[i] = ps.ss[i]->conv[il];
        sg.ssm[i] = ps.ss[i]->ssm[il];
        sg.kc[i] = ps.ss[i]->kc[il];
        sg.vc[i] = ps.ss[i]->vc[il];
    }
    sg.col0[ps.n] = ps.col0[ps.n];
    sg.pos0 = ps.pos_dev;
    return sg;
}

// lm: the pass ends in the output norm of its (at most kSmallBatch) columns for
// run_lmhead_batch, each column's stream stored to its state.
int run_pass(const qg_model* m, const Pass& ps, Scratch* sc, cudaStream_t st, bool lm = false) {
    const qg_config& c = m->cfg;
    const int H = c.hidden, P = ps.col0[ps.n];
    const bool small = P <= kSmallBatch;    // a batched decode step: the small-batch GEMV
    const int ldk = !small ? kPfChunk : P <= 4 ? 4 : 8;  // stride of the gate/up outputs, k-major
    const int ldin = small ? ldk : 0;       // GEMM inputs: packed [k][4] or [k][8] columns, or the tensor-core tiles
    const size_t part = static_cast<size_t>(P) * H;
    const bool kvq = ps.ss[0]->kv_format == QG_KV_Q8_0_Q5_1;
    unsigned* err = ps.ss[0]->err;  // the small-batch GEMV's bounded waits report here
    const bool pdl = small;         // programmatic chaining of the pass's kernels: a batched decode step only
    if (int e_ = launch_pdl(pf_embed_kernel, dim3(P), dim3(256), 0, st, pdl, m->embd, sc->tok, H, sc->X))
        return e_;
    int pending = 0;  // split sums of the last projection not yet added to X
    int rc = QG_OK;
    for (int il = 0; il < c.n_layers && !rc; ++il) {
        const qg_layer_dev& L = m->layers[il];
        const Segs sg = segs_of(ps, il);
        if (int e_ = add_norm(P, pdl, st, sc->X, sc->Yp, pending, part, L.attn_norm, sc->Xn, ldin, H, c.eps, HOut{}))
            return e_;
        int zin = 1;
        if ((rc = gemm<QT_Q4K, false>(L.w_in, L.n_in, H, sc->Xn, sc->Zp, L.n_in, P, splits_for(L.n_in, H, P), st, &zin,
                                      err, sc->cap_zp)))
            break;
        const float* Z = sc->Zp;  // the input projection's output [P][n_in]: one split is already the sum
        if (zin > 1) {
            const size_t cnt = static_cast<size_t>(P) * L.n_in;
            if (int e_ = launch_pdl(pf_sum_parts_kernel, dim3(static_cast<unsigned>((cnt + 255) / 256)), dim3(256), 0,
                                    st, pdl, sc->Zp, zin, cnt, sc->Z, cnt))
                return e_;
            Z = sc->Z;
        }
        int k_out;
        if (m->kinds[il] == QG_LAYER_DELTANET) {
            const int C = m->conv_dim, nv = c.n_v_heads, dv = c.head_v_dim;
            const long long cg = static_cast<long long>(P) * (C + nv);
            if (ps.n == 1 && c.conv_kernel == 4 && P > kSmallBatch) {  // one sequence's prompt chunk
                if (int e_ = launch_pdl(pf_conv4_block_kernel,
                                        dim3(static_cast<unsigned>((C + nv + 255) / 256), (P + kConvTB - 1) / kConvTB),
                                        dim3(256), 0, st, pdl, Z, L.n_in, P, C, nv, sg.conv[0], L.conv_w, L.dt_bias,
                                        L.a, sc->Cq, sc->dt, sc->beta))
                    return e_;
            } else if (int e_ = launch_pdl(pf_conv_gates_kernel, dim3(static_cast<unsigned>((cg + 255) / 256)),
                                           dim3(256), 0, st, pdl, Z, L.n_in, P, C, nv, c.conv_kernel, sg, L.conv_w,
                                           L.dt_bias, L.a, sc->Cq, sc->dt, sc->beta)) {
                return e_;
            }
            if (int e_ = launch_pdl(pf_conv_window_kernel, dim3((C + 255) / 256, ps.n), dim3(256), 0, st, pdl, Z,
                                    L.n_in, C, c.conv_kernel, sg))
                return e_;
            const int warps = P * 2 * c.n_k_heads;
            if (int e_ = launch_pdl(pf_l2norm_kernel, dim3((warps * 32 + 255) / 256), dim3(256), 0, st, pdl, sc->Cq, C,
                                    m->k_dim, c.n_k_heads, P, c.eps, sc->QKn))
                return e_;
            if (int e_ = launch_pdl(pf_delta_kernel, dim3(nv * dv / 32, ps.n), dim3(256), 0, st, pdl, sc->Cq, C,
                                    m->k_dim, sc->QKn, sc->dt, sc->beta, sg, sc->O, c.n_k_heads, nv, dv))
                return e_;
            if (int e_ = launch_pdl(pf_gated_norm_kernel, dim3(P, (nv + 7) / 8), dim3(256), 0, st, pdl, sc->O, Z,
                                    L.n_in, C + 2 * nv, L.ssm_norm, nv, dv, c.eps, sc->Uin, ldin))
                return e_;
            k_out = m->v_dim;
        } else {
            const int nkv = c.n_kv_heads, kvd = m->kv_dim;
            if (int e_ = launch_pdl(pf_attn_prep_kernel, dim3(P), dim3(256), 0, st, pdl, Z, L.n_in, c.n_heads, nkv,
                                    L.q_norm, L.k_norm, sg, c.n_rot, m->theta_scale, c.eps, sc->Qn,
                                    kvq ? sc->Ks : nullptr, kvq ? sc->Vs : nullptr))
                return e_;
            for (int i = 0; kvq && i < ps.n && !rc; ++i) {
                const qg_state* si = ps.ss[i];
                const size_t off = static_cast<size_t>(ps.col0[i]) * kvd;
                rc = kv_quantize_rows_dev(sc->Ks + off, sc->Vs + off, ps.col0[i + 1] - ps.col0[i], ps.pos_dev + i,
                                          nkv, si->max_seq, reinterpret_cast<uint8_t*>(si->kc[il]),
                                          reinterpret_cast<uint8_t*>(si->vc[il]), st);
            }
            if (rc) break;
            const int gs = c.n_heads / nkv;
            const int zs = pdl ? kAttnSplits : 1;  // a batched decode step: key splits, then a merge
            float* part = zs > 1 ? sc->Ap : nullptr;
            const dim3 grid(P, nkv, zs);
            rc = kvq ? launch_causal<true>(gs, grid, st, pdl, sc->Qn, Z, L.n_in, sg, kvd, sc->Uin, ldin, part)
                     : launch_causal<false>(gs, grid, st, pdl, sc->Qn, Z, L.n_in, sg, kvd, sc->Uin, ldin, part);
            if (rc) break;
            if (part) {
                if (int e_ = launch_pdl(pf_attn_merge_kernel, dim3(P, c.n_heads), dim3(kHd), 0, st, pdl, part, zs, Z,
                                        L.n_in, sc->Uin, ldin))
                    return e_;
            }
            k_out = m->q_dim;
        }
        if ((rc = gemm<QT_Q4K, false>(L.w_out, H, k_out, sc->Uin, sc->Yp, H, P, splits_for(H, k_out, P), st, &pending,
                                      err, sc->cap_yp)))
            break;
        if (int e_ = add_norm(P, pdl, st, sc->X, sc->Yp, pending, part, L.post_norm, sc->Xn, ldin, H, c.eps, HOut{}))
            return e_;
        const int zf = splits_for(c.ffn, H, P);
        int zg = 1, zu = 1;
        if (small) {  // row-major [ffn][ldk] sums for the small-batch SwiGLU
            if ((rc = gemm<QT_Q4K, true>(L.w_gate, c.ffn, H, sc->Xn, sc->Zp, ldk, P, zf, st, &zg, err, sc->cap_zp))) break;
            if ((rc = gemm<QT_Q4K, true>(L.w_up, c.ffn, H, sc->Xn, sc->Up, ldk, P, zf, st, &zu, err, sc->cap_up))) break;
        } else {  // token-major [P][ffn]
            if ((rc = gemm<QT_Q4K, false>(L.w_gate, c.ffn, H, sc->Xn, sc->Zp, c.ffn, P, zf, st, &zg, err, sc->cap_zp))) break;
            if ((rc = gemm<QT_Q4K, false>(L.w_up, c.ffn, H, sc->Xn, sc->Up, c.ffn, P, zf, st, &zu, err, sc->cap_up))) break;
        }
        const size_t na = static_cast<size_t>(c.ffn) * P;  // ffn values of each of the P columns
        if (int e_ = launch_pdl(pf_swiglu_kernel, dim3(static_cast<unsigned>((na + 255) / 256)), dim3(256), 0, st, pdl,
                                sc->Zp, zg, sc->Up, zu, static_cast<size_t>(c.ffn) * (small ? ldk : P), sc->A, c.ffn,
                                P, small ? ldk : 0, ldin))
            return e_;
        rc = gemm<QT_Q6K, false>(L.w_down, H, c.ffn, sc->A, sc->Yp, H, P, splits_for(H, c.ffn, P), st, &pending, err,
                        sc->cap_yp);
    }
    if (rc) return rc;
    if (lm) {  // batched lm_head next: the output norm of every column, each stream to its state
        HOut ho{};
        for (int i = 0; i < ps.n; ++i) ho.h[i] = ps.ss[i]->h;
        return add_norm(P, pdl, st, sc->X, sc->Yp, pending, part, m->out_norm, sc->Xn, ldin, H, c.eps, ho);
    }
    return add_norm(P, pdl, st, sc->X, sc->Yp, pending, part, nullptr, nullptr, kPfChunk, H, c.eps, HOut{});
}

// The lm_head argmax of every column of a batched pass (at most kSmallBatch,
// after run_pass with lm): one small-batch GEMV per 4 columns over the
// output-normed columns in sc->Xn, each column's token into its sequence's
// slots, masked by its sequence's allow bitset.
int run_lmhead_batch(const qg_model* m, const Pass& ps, Scratch* sc, cudaStream_t st) {
    const int xq = ps.n <= 4 ? 4 : 8;
    for (int g = 0; 4 * g < ps.n; ++g) {
        BmArgmax am{};
        const int nm = std::min(4, ps.n - 4 * g);
        for (int c = 0; c < nm; ++c) {
            const qg_state* si = ps.ss[4 * g + c];
            am.ws[c] = si->am_ws;
            am.slots[c] = si->slots;
            am.allow[c] = si->allow;
            am.err[c] = si->err;
        }
        if (int rc = launch_bm4<QT_Q6K, false, true>(m->lm_head, m->cfg.vocab, m->cfg.hidden, sc->Xn + 4 * g, xq,
                                                     nullptr, 0, 0, nm, am, ps.ss[0]->err, st, nullptr))
            return rc;
    }
    return QG_OK;
}

}  // namespace

void prefill_release(qg_state* s) {  // the device buffers belong to s->allocs
    delete static_cast<Scratch*>(s->pf);
    s->pf = nullptr;
}

}  // namespace qg

using namespace qg;

extern "C" int qg_prefill(qg_model* m, qg_state* s, const uint32_t* tokens, int n_tokens, int pos0,
                          uint32_t* next_token) {
    if (!m || !s || !next_token) return set_err(QG_ERR_ARG, "prefill: NULL argument");
    if (s->m != m) return set_err(QG_ERR_ARG, "prefill: state belongs to another model");
    if (n_tokens < 1) return set_err(QG_ERR_SHAPE, "prefill: %d tokens", n_tokens);
    if (!tokens) return set_err(QG_ERR_ARG, "prefill: NULL tokens");
    if (pos0 < 0 || pos0 + n_tokens > s->max_seq)
        return set_err(QG_ERR_POS, "prefill: positions %d..%d are past the KV cache (%d rows)", pos0,
                       pos0 + n_tokens - 1, s->max_seq);
    const qg_config& c = m->cfg;
    for (int i = 0; i < n_tokens; ++i)
        if (tokens[i] >= static_cast<uint32_t>(c.vocab))
            return set_err(QG_ERR_TOKEN, "prefill: token %u is outside the %d-row embedding table", tokens[i], c.vocab);
    if (c.head_k_dim != kDk) return set_err(QG_ERR_SHAPE, "prefill: head_k_dim %d is not served", c.head_k_dim);
    DeviceGuard dg(m->device);
    Scratch* sc = nullptr;
    int rc = scratch_of(m, s, &sc);
    if (rc) return rc;
    cudaStream_t st = s->stream;
    QG_CUDA(cudaStreamSynchronize(st));
    for (int c0 = 0; c0 < n_tokens && !rc; c0 += sc->chunk) {
        const int P = std::min(sc->chunk, n_tokens - c0);
        QG_CUDA(cudaMemcpyAsync(sc->tok, tokens + c0, sizeof(int) * P, cudaMemcpyHostToDevice, st));
        const int p0 = pos0 + c0;
        QG_CUDA(cudaMemcpyAsync(sc->pos, &p0, sizeof(int), cudaMemcpyHostToDevice, st));
        QG_CUDA(cudaStreamSynchronize(st));  // p0 lives on this frame
        Pass ps{};
        ps.n = 1;
        ps.ss[0] = s;
        ps.pos_dev = sc->pos;
        ps.col0[0] = 0;
        ps.col0[1] = P;
        rc = run_pass(m, ps, sc, st);
        if (!rc && c0 + P >= n_tokens)
            rc = run_lmhead_of(m, s, sc->X + static_cast<size_t>(P - 1) * c.hidden, st);
        if (!rc) QG_CUDA(cudaStreamSynchronize(st));  // the token copy of the next chunk reuses sc->tok
    }
    if (rc) return rc;
    unsigned out = 0;
    QG_CUDA(cudaMemcpy(&out, s->slots + 2, sizeof out, cudaMemcpyDeviceToHost));
    if (out & 0x80000000u) {
        unsigned e = 0;
        cudaMemcpy(&e, s->err, sizeof e, cudaMemcpyDeviceToHost);
        return set_err(QG_ERR_TIMEOUT, "prefill: a kernel gave up on a bounded wait (flags 0x%x)", e);
    }
    *next_token = out;
    if (s->kv_len < pos0 + n_tokens) s->kv_len = pos0 + n_tokens;
    return QG_OK;
}

extern "C" int qg_decode_batch(qg_model* m, qg_state* const* states, int n, const uint32_t* tokens,
                               const int* positions, uint32_t* next_tokens) {
    if (!m || !states || !tokens || !positions || !next_tokens) return set_err(QG_ERR_ARG, "decode_batch: NULL argument");
    if (n < 1 || n > kMaxSeg) return set_err(QG_ERR_SHAPE, "decode_batch: %d sequences (served: 1..%d)", n, kMaxSeg);
    const qg_config& c = m->cfg;
    if (c.head_k_dim != kDk) return set_err(QG_ERR_SHAPE, "decode_batch: head_k_dim %d is not served", c.head_k_dim);
    for (int i = 0; i < n; ++i) {
        qg_state* si = states[i];
        if (!si || si->m != m) return set_err(QG_ERR_ARG, "decode_batch: state %d is NULL or of another model", i);
        if (si->kv_format != states[0]->kv_format)
            return set_err(QG_ERR_ARG, "decode_batch: the states' KV cache formats differ");
        for (int j = 0; j < i; ++j)
            if (states[j] == si) return set_err(QG_ERR_ARG, "decode_batch: state %d appears twice", i);
        if (tokens[i] >= static_cast<uint32_t>(c.vocab))
            return set_err(QG_ERR_TOKEN, "decode_batch: token %u is outside the %d-row embedding table", tokens[i], c.vocab);
        if (positions[i] < 0 || positions[i] >= si->max_seq)
            return set_err(QG_ERR_POS, "decode_batch: position %d is past the KV cache (%d rows)", positions[i], si->max_seq);
    }
    DeviceGuard dg(m->device);
    Scratch* sc = nullptr;
    int rc = scratch_of(m, states[0], &sc);
    if (rc) return rc;
    for (int i = 0; i < n; ++i) QG_CUDA(cudaStreamSynchronize(states[i]->stream));
    cudaStream_t st = states[0]->stream;
    QG_CUDA(cudaMemcpyAsync(sc->tok, tokens, sizeof(int) * n, cudaMemcpyHostToDevice, st));
    QG_CUDA(cudaMemcpyAsync(sc->pos, positions, sizeof(int) * n, cudaMemcpyHostToDevice, st));
    Pass ps{};
    ps.n = n;
    ps.pos_dev = sc->pos;
    for (int i = 0; i < n; ++i) {
        ps.ss[i] = states[i];
        ps.col0[i] = i;
    }
    ps.col0[n] = n;
    const bool lmb = n <= kSmallBatch;  // batched lm_head launches, one per 4 sequences
    rc = run_pass(m, ps, sc, st, lmb);
    if (!rc && lmb) rc = run_lmhead_batch(m, ps, sc, st);
    for (int i = 0; i < n && !rc && !lmb; ++i)
        rc = run_lmhead_of(m, states[i], sc->X + static_cast<size_t>(i) * c.hidden, st);
    if (rc) return rc;
    QG_CUDA(cudaStreamSynchronize(st));
    for (int i = 0; i < n; ++i) {
        unsigned out = 0;
        QG_CUDA(cudaMemcpy(&out, states[i]->slots + 2, sizeof out, cudaMemcpyDeviceToHost));
        if (out & 0x80000000u) {
            unsigned e = 0;
            cudaMemcpy(&e, states[i]->err, sizeof e, cudaMemcpyDeviceToHost);
            return set_err(QG_ERR_TIMEOUT, "decode_batch: a kernel gave up on a bounded wait (flags 0x%x)", e);
        }
        next_tokens[i] = out;
        if (states[i]->kv_len < positions[i] + 1) states[i]->kv_len = positions[i] + 1;
    }
    return QG_OK;
}

// ----------------------------------------------------------- batch graphs
// A fixed set of sequences decoded in lockstep through one captured CUDA graph:
// per step, the tokens and positions go in from pinned host memory, the pass
// and each sequence's lm_head argmax run, and the n token words come back.
struct qg_batch {
    qg_model* m;
    int n;
    qg_state* ss[kMaxSeg];
    int* pinned;  // [0, 16) tokens, [16, 32) positions, [32, 48) token words out
    cudaGraphExec_t exec;
};

namespace {

int batch_check(const qg_model* m, qg_state* const* states, int n) {
    if (n < 1 || n > kMaxSeg) return set_err(QG_ERR_SHAPE, "batch: %d sequences (served: 1..%d)", n, kMaxSeg);
    if (m->cfg.head_k_dim != kDk) return set_err(QG_ERR_SHAPE, "batch: head_k_dim %d is not served", m->cfg.head_k_dim);
    for (int i = 0; i < n; ++i) {
        qg_state* si = states[i];
        if (!si || si->m != m) return set_err(QG_ERR_ARG, "batch: state %d is NULL or of another model", i);
        if (si->kv_format != states[0]->kv_format) return set_err(QG_ERR_ARG, "batch: the states' KV cache formats differ");
        for (int j = 0; j < i; ++j)
            if (states[j] == si) return set_err(QG_ERR_ARG, "batch: state %d appears twice", i);
    }
    return QG_OK;
}

int batch_inputs_check(const qg_model* m, qg_state* const* states, int n, const uint32_t* tokens,
                       const int* positions) {
    for (int i = 0; i < n; ++i) {
        if (tokens[i] >= static_cast<uint32_t>(m->cfg.vocab))
            return set_err(QG_ERR_TOKEN, "batch: token %u is outside the %d-row embedding table", tokens[i], m->cfg.vocab);
        if (positions[i] < 0 || positions[i] >= states[i]->max_seq)
            return set_err(QG_ERR_POS, "batch: position %d is past the KV cache (%d rows)", positions[i],
                           states[i]->max_seq);
    }
    return QG_OK;
}

}  // namespace

extern "C" int qg_batch_create(qg_model* m, qg_state* const* states, int n, qg_batch** out) {
    if (!m || !states || !out) return set_err(QG_ERR_ARG, "batch_create: NULL argument");
    int rc = batch_check(m, states, n);
    if (rc) return rc;
    DeviceGuard dg(m->device);
    Scratch* sc = nullptr;
    if ((rc = scratch_of(m, states[0], &sc))) return rc;
    qg_batch* b = new (std::nothrow) qg_batch();
    if (!b) return set_err(QG_ERR_OOM, "batch_create: host allocation");
    b->m = m;
    b->n = n;
    for (int i = 0; i < n; ++i) b->ss[i] = states[i];
    b->exec = nullptr;
    void* p = nullptr;
    const cudaError_t e = cudaHostAlloc(&p, 48 * sizeof(int), cudaHostAllocDefault);
    if (e != cudaSuccess) {
        delete b;
        return cuda_err(e, "batch_create: cudaHostAlloc");
    }
    b->pinned = static_cast<int*>(p);
    std::memset(b->pinned, 0, 48 * sizeof(int));
    *out = b;
    return QG_OK;
}

extern "C" int qg_batch_destroy(qg_batch* b) {
    if (!b) return QG_OK;
    DeviceGuard dg(b->m->device);
    cudaStreamSynchronize(b->ss[0]->stream);
    if (b->exec) cudaGraphExecDestroy(b->exec);
    if (b->pinned) cudaFreeHost(b->pinned);
    delete b;
    return QG_OK;
}

extern "C" int qg_batch_step(qg_batch* b, const uint32_t* tokens, const int* positions, uint32_t* next_tokens) {
    if (!b || !tokens || !positions || !next_tokens) return set_err(QG_ERR_ARG, "batch_step: NULL argument");
    qg_model* m = b->m;
    const int n = b->n;
    int rc = batch_inputs_check(m, b->ss, n, tokens, positions);
    if (rc) return rc;
    DeviceGuard dg(m->device);
    for (int i = 1; i < n; ++i) QG_CUDA(cudaStreamSynchronize(b->ss[i]->stream));
    cudaStream_t st = b->ss[0]->stream;
    QG_CUDA(cudaStreamSynchronize(st));
    Scratch* sc = static_cast<Scratch*>(b->ss[0]->pf);
    for (int i = 0; i < n; ++i) {
        b->pinned[i] = static_cast<int>(tokens[i]);
        b->pinned[16 + i] = positions[i];
    }
    if (!b->exec) {  // capture once: copies in, the pass, each lm_head, the token words out
        cudaGraph_t g = nullptr;
        QG_CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeRelaxed));
        cudaError_t e = cudaMemcpyAsync(sc->tok, b->pinned, sizeof(int) * n, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(sc->pos, b->pinned + 16, sizeof(int) * n, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) rc = cuda_err(e, "batch_step: capture H2D");
        Pass ps{};
        ps.n = n;
        ps.pos_dev = sc->pos;
        for (int i = 0; i < n; ++i) {
            ps.ss[i] = b->ss[i];
            ps.col0[i] = i;
        }
        ps.col0[n] = n;
        const bool lmb = n <= kSmallBatch;  // batched lm_head launches, one per 4 sequences
        if (!rc) rc = run_pass(m, ps, sc, st, lmb);
        if (!rc && lmb) rc = run_lmhead_batch(m, ps, sc, st);
        for (int i = 0; i < n && !rc && !lmb; ++i)
            rc = run_lmhead_of(m, b->ss[i], sc->X + static_cast<size_t>(i) * m->cfg.hidden, st);
        for (int i = 0; i < n && !rc; ++i) {
            e = cudaMemcpyAsync(b->pinned + 32 + i, b->ss[i]->slots + 2, sizeof(int), cudaMemcpyDeviceToHost, st);
            if (e != cudaSuccess) rc = cuda_err(e, "batch_step: capture D2H");
        }
        const cudaError_t ee = cudaStreamEndCapture(st, &g);
        if (!rc && ee != cudaSuccess) rc = cuda_err(ee, "batch_step: cudaStreamEndCapture");
        if (!rc) {
            e = cudaGraphInstantiate(&b->exec, g, 0);
            if (e != cudaSuccess) {
                rc = cuda_err(e, "batch_step: cudaGraphInstantiate");
                b->exec = nullptr;
            }
        }
        if (g) cudaGraphDestroy(g);
        if (rc) return rc;
    }
    QG_CUDA(cudaGraphLaunch(b->exec, st));
    QG_CUDA(cudaStreamSynchronize(st));
    for (int i = 0; i < n; ++i) {
        const unsigned w = static_cast<unsigned>(b->pinned[32 + i]);
        if (w & 0x80000000u) {
            unsigned e = 0;
            cudaMemcpy(&e, b->ss[i]->err, sizeof e, cudaMemcpyDeviceToHost);
            return set_err(QG_ERR_TIMEOUT, "batch_step: a kernel gave up on a bounded wait (flags 0x%x)", e);
        }
        next_tokens[i] = w;
        if (b->ss[i]->kv_len < positions[i] + 1) b->ss[i]->kv_len = positions[i] + 1;
    }
    return QG_OK;
}
