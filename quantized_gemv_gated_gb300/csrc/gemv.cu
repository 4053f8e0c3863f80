// Building-block entry points: Q4_K GEMV, planar Q4_K / Q6_K GEMV and repacks, the
// fused lm_head GEMV + argmax and a plain argmax; plus the error plumbing
// shared by the whole library.
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "qg_host.cuh"

namespace qg {

static thread_local char g_msg[512];

int set_err(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_err(cudaError_t e, const char* what) {
    return set_err(e == cudaErrorMemoryAllocation ? QG_ERR_OOM : QG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int device_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    static std::atomic<int> cache[64];  // zero-initialised; a racing first call stores the same value
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c) return c;
    }
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (v < 1) v = 1;
    if (dev >= 0 && dev < 64) cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

int grant_smem(const void* kern, int smem) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> granted;  // (kernel, device) -> bytes
    int dev = 0;
    QG_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lock(mu);
    int& have = granted[std::make_pair(kern, dev)];
    if (smem > have) {
        QG_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        QG_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     static_cast<int>(cudaSharedmemCarveoutMaxShared)));
        have = smem;
    }
    return QG_OK;
}

// Error word of the building blocks (one per device that loads the library).
__device__ unsigned g_block_err;

static unsigned* block_err_ptr() {
    static std::mutex mu;
    static unsigned* cache[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        unsigned* p = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_block_err) != cudaSuccess) return nullptr;
        cache[dev] = p;
    }
    return cache[dev];
}

// Static scratch of qg_lmhead_argmax_noalloc: the fused argmax's workspace
// (best key, arrival count), 16 of its 256 bytes in use.  A __device__ array
// without an initializer is zero when the module loads, and every call leaves
// it zeroed again (the last CTA clears it), so no call needs to clear it first.
static __device__ __align__(256) unsigned long long g_lmhead_scratch[32];

static int lmhead_scratch(unsigned long long** out) {
    static std::mutex mu;
    static unsigned long long* cache[64] = {nullptr};
    int dev = 0;
    QG_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return set_err(QG_ERR_ARG, "lmhead_argmax_noalloc: device %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        unsigned long long* p = nullptr;
        QG_CUDA(cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_lmhead_scratch));
        cache[dev] = p;
    }
    *out = cache[dev];
    return QG_OK;
}

// ------------------------------------------------- grouped weight layouts
// One thread per (8-row group, super-block) of the padded matrix, stored at
// its slice-major place (grouped_offset); rows n..n8-1 are zero.  Q6_K: for
// row rr and quarter cq = 2 half + part (u = 4 rr + cq) the 48-byte record
// [ql[64 half + 16 part ..16] | ql[64 half + 32 + 16 part ..16] | qh[16 cq ..16]]
// at 48u, the quarter's scales sc[8 half + part + 2s] (s = 0..3) at 1536 + 4u,
// d at 1664 + 2 rr.  Q4_K: the 8 rows' 144-byte blocks.
__global__ void q6k_grouped_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int n, int n8, int nb) {
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long total = static_cast<long long>(n8 / 8) * nb;
    if (idx >= total) return;
    const long long g = idx / nb, b = idx - g * nb;
    uint8_t* gb = dst + grouped_offset(n8, nb, static_cast<int>(g), static_cast<int>(b), 1680);
    for (int rr = 0; rr < 8; ++rr) {
        const long long r = 8 * g + rr;
        const uint8_t* blk = r < n ? src + (r * nb + b) * 210 : nullptr;
        for (int cq = 0; cq < 4; ++cq) {
            const int half = cq >> 1, part = cq & 1, u = 4 * rr + cq;
            uint8_t* rec = gb + 48 * u;
            uint8_t* sc = gb + 1536 + 4 * u;
            for (int i = 0; i < 16; ++i) {
                rec[i] = blk ? blk[64 * half + 16 * part + i] : 0;
                rec[16 + i] = blk ? blk[64 * half + 32 + 16 * part + i] : 0;
                rec[32 + i] = blk ? blk[128 + 16 * cq + i] : 0;
            }
            for (int s = 0; s < 4; ++s) sc[s] = blk ? blk[192 + 8 * half + part + 2 * s] : 0;
        }
        gb[1664 + 2 * rr] = blk ? blk[208] : 0;
        gb[1665 + 2 * rr] = blk ? blk[209] : 0;
    }
}

__global__ void q4k_grouped_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int n, int n8, int nb) {
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long total = static_cast<long long>(n8 / 8) * nb;
    if (idx >= total) return;
    const long long g = idx / nb, b = idx - g * nb;
    uint4* gb = reinterpret_cast<uint4*>(dst + grouped_offset(n8, nb, static_cast<int>(g), static_cast<int>(b), 1152));
    for (int rr = 0; rr < 8; ++rr) {
        const long long r = 8 * g + rr;
        for (int i = 0; i < 9; ++i)
            gb[rr * 9 + i] = r < n ? reinterpret_cast<const uint4*>(src + (r * nb + b) * 144)[i] : make_uint4(0u, 0u, 0u, 0u);
    }
}

int q4k_to_grouped(const void* src, void* dst, int n, int k, cudaStream_t st) {
    const int nb = k / 256, n8 = (n + 7) & ~7;
    const long long total = static_cast<long long>(n8 / 8) * nb;
    const long long blocks = (total + 255) / 256;
    q4k_grouped_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const uint8_t*>(src),
                                                                     static_cast<uint8_t*>(dst), n, n8, nb);
    QG_CUDA(cudaGetLastError());
    return QG_OK;
}

int q6k_to_planar(const void* src, void* dst, int n, int k, cudaStream_t st) {
    const int nb = k / 256, n8 = (n + 7) & ~7;
    const long long total = static_cast<long long>(n8 / 8) * nb;
    const long long blocks = (total + 255) / 256;
    q6k_grouped_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const uint8_t*>(src),
                                                                     static_cast<uint8_t*>(dst), n, n8, nb);
    QG_CUDA(cudaGetLastError());
    return QG_OK;
}

// -------------------------------------------------------------- argmax f32
__global__ void __launch_bounds__(1024) argmax_f32_kernel(const float* __restrict__ x, int n, uint32_t* out) {
    __shared__ unsigned long long red[32];
    unsigned long long best = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const unsigned long long key = argmax_key(__ldcg(x + i), static_cast<unsigned>(i));
        best = key > best ? key : best;
    }
    best = warp_max_u64(best);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x < 32) {
        unsigned long long v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0ull;
        v = warp_max_u64(v);
        if (threadIdx.x == 0) *out = v ? argmax_key_index(v) : 0u;
    }
}

// ------------------------------------------------- lm_head GEMV + argmax epilogue
// Per-row keys reduce to one per CTA, CTAs combine with a 64-bit atomicMax
// (max is exact, so the result does not depend on arrival order), and the
// last CTA to arrive publishes the token and re-zeroes the workspace.
struct EpiArgmax : EpiBase {
    unsigned long long* ws;  // ws[0]: best key; ws[1] low word: arrivals
    uint32_t* tok;
    unsigned long long best;
    __device__ void start() { best = 0ull; }
    __device__ void apply(int r0, int r1, const float* ys, const float*, int tid) {
        for (int r = r0 + tid; r < r1; r += kConsumers) {
            const unsigned long long key = argmax_key(ys[r - r0], static_cast<unsigned>(r));
            best = key > best ? key : best;
        }
    }
    __device__ void finish(float* sm, int tid) {
        unsigned long long* red = reinterpret_cast<unsigned long long*>(sm);
        best = warp_max_u64(best);
        if ((tid & 31) == 0) red[tid >> 5] = best;
        bar_sync(1, kConsumers);
        if (tid == 0) {
            unsigned long long m = 0ull;
            for (int i = 0; i < kConsumerWarps; ++i) m = red[i] > m ? red[i] : m;
            atomicMax(ws, m);
            __threadfence();
            const unsigned prev = atomicAdd(reinterpret_cast<unsigned*>(ws + 1), 1u);
            if (prev == gridDim.x - 1) {
                __threadfence();
                const unsigned long long key = atomicExch(ws, 0ull);
                atomicExch(reinterpret_cast<unsigned*>(ws + 1), 0u);
                *tok = key ? argmax_key_index(key) : 0u;
            }
        }
    }
};

}  // namespace qg

using namespace qg;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// y (an f32 vector, or the 4-byte token slot of the fused argmax) is written
// with 4-byte stores: a misaligned pointer is refused here, before any launch.
static int check_gemv_args(const void* w, const float* x, const void* y, int n, int k) {
    if (!w || !x || !y) return set_err(QG_ERR_ARG, "gemv: NULL pointer");
    if (n < 0 || k < 0) return set_err(QG_ERR_ARG, "gemv: negative size n=%d k=%d", n, k);
    if (n == 0 || k == 0) return set_err(QG_ERR_EMPTY, "gemv: empty tensor n=%d k=%d", n, k);
    if (!gemv_k_served(k)) return set_err(QG_ERR_SHAPE, "gemv: k=%d is not a multiple of 256 up to 16384", k);
    if (!aligned16(w) || !aligned16(x)) return set_err(QG_ERR_ARG, "gemv: w and x must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(y) & 3u) return set_err(QG_ERR_ARG, "gemv: y / tok_dev must be 4-byte aligned");
    return QG_OK;
}

extern "C" {

const char* qg_last_error(void) { return g_msg; }

int qg_gemv_q4k(const void* w, const float* x, float* y, int n, int k, qg_stream stream) {
    int rc = check_gemv_args(w, x, y, n, k);
    if (rc) return rc;
    EpiStore epi{};
    epi.y = y;
    return launch_gemv<QT_Q4K, false, LAYOUT_RAW>(w, nullptr, n, k, ProPlainG{x}, epi,
                                                  reinterpret_cast<cudaStream_t>(stream), true, block_err_ptr());
}

int qg_gemv_q6k_planar(const void* w_planar, const float* x, float* y, int n, int k, qg_stream stream) {
    int rc = check_gemv_args(w_planar, x, y, n, k);
    if (rc) return rc;
    EpiStore epi{};
    epi.y = y;
    return launch_gemv<QT_Q6K, false>(w_planar, nullptr, n, k, ProPlainG{x}, epi,
                                      reinterpret_cast<cudaStream_t>(stream), true, block_err_ptr());
}

int qg_gemv_q4k_planar(const void* w_planar, const float* x, float* y, int n, int k, qg_stream stream) {
    int rc = check_gemv_args(w_planar, x, y, n, k);
    if (rc) return rc;
    EpiStore epi{};
    epi.y = y;
    return launch_gemv<QT_Q4K, false>(w_planar, nullptr, n, k, ProPlainG{x}, epi,
                                      reinterpret_cast<cudaStream_t>(stream), true, block_err_ptr());
}

size_t qg_q4k_planar_bytes(int n, int k) {
    if (n <= 0 || k <= 0 || k % 256) return 0;
    return static_cast<size_t>((n + 7) & ~7) * (k / 256) * 144;
}

int qg_q4k_to_planar(const void* src, void* dst, int n, int k, qg_stream stream) {
    if (!src || !dst) return set_err(QG_ERR_ARG, "q4k_to_planar: NULL pointer");
    if (n <= 0 || k <= 0) return set_err(QG_ERR_EMPTY, "q4k_to_planar: empty tensor n=%d k=%d", n, k);
    if (k % 256) return set_err(QG_ERR_SHAPE, "q4k_to_planar: k=%d is not a multiple of 256", k);
    if (!aligned16(dst)) return set_err(QG_ERR_ARG, "q4k_to_planar: dst must be 16-byte aligned");
    return q4k_to_grouped(src, dst, n, k, reinterpret_cast<cudaStream_t>(stream));
}

size_t qg_q6k_planar_bytes(int n, int k) {
    if (n <= 0 || k <= 0 || k % 256) return 0;
    return static_cast<size_t>((n + 7) & ~7) * (k / 256) * 210;
}

int qg_q6k_to_planar(const void* src, void* dst, int n, int k, qg_stream stream) {
    if (!src || !dst) return set_err(QG_ERR_ARG, "q6k_to_planar: NULL pointer");
    if (n <= 0 || k <= 0) return set_err(QG_ERR_EMPTY, "q6k_to_planar: empty tensor n=%d k=%d", n, k);
    if (k % 256) return set_err(QG_ERR_SHAPE, "q6k_to_planar: k=%d is not a multiple of 256", k);
    if (!aligned16(dst)) return set_err(QG_ERR_ARG, "q6k_to_planar: dst must be 16-byte aligned");
    return q6k_to_planar(src, dst, n, k, reinterpret_cast<cudaStream_t>(stream));
}

size_t qg_lmhead_argmax_workspace_bytes(void) { return 16; }

int qg_lmhead_argmax(const void* w_planar, const float* x, int n_vocab, int k, void* workspace, uint32_t* tok_dev,
                     qg_stream stream) {
    int rc = check_gemv_args(w_planar, x, tok_dev, n_vocab, k);
    if (rc) return rc;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 7u))
        return set_err(QG_ERR_ARG, "lmhead_argmax: workspace must be 8-byte aligned device memory");
    EpiArgmax epi{};
    epi.ws = static_cast<unsigned long long*>(workspace);
    epi.tok = tok_dev;
    return launch_gemv<QT_Q6K, false>(w_planar, nullptr, n_vocab, k, ProPlainG{x}, epi,
                                      reinterpret_cast<cudaStream_t>(stream), true, block_err_ptr());
}

// The same GEMV + argmax with its workspace in static device memory, for
// callers that must not allocate: a process whose device memory is reserved up
// front by a pool (a cudaMalloc there fails or evicts the pool), or a decode
// loop on a latency budget, where an allocation call can synchronise the
// device.  Nothing here calls cudaMalloc / cudaFree or an allocating library
// routine; the first call on a device resolves the scratch address with
// cudaGetSymbolAddress (nothing is copied or synchronised), later calls only
// launch.
int qg_lmhead_argmax_noalloc(const void* w_planar, const float* x, int n_vocab, int k, uint32_t* tok_dev,
                             qg_stream stream) {
    int rc = check_gemv_args(w_planar, x, tok_dev, n_vocab, k);
    if (rc) return rc;
    if (qg_lmhead_argmax_workspace_bytes() > sizeof(g_lmhead_scratch))
        return set_err(QG_ERR_SHAPE, "lmhead_argmax_noalloc: the kernel needs %zu bytes of scratch, the static area "
                                     "holds %zu", qg_lmhead_argmax_workspace_bytes(), sizeof(g_lmhead_scratch));
    unsigned long long* ws = nullptr;
    rc = lmhead_scratch(&ws);
    if (rc) return rc;
    EpiArgmax epi{};
    epi.ws = ws;
    epi.tok = tok_dev;
    return launch_gemv<QT_Q6K, false>(w_planar, nullptr, n_vocab, k, ProPlainG{x}, epi,
                                      reinterpret_cast<cudaStream_t>(stream), true, block_err_ptr());
}

int qg_argmax_f32(const float* x, int n, uint32_t* idx_dev, qg_stream stream) {
    if (!x || !idx_dev) return set_err(QG_ERR_ARG, "argmax_f32: NULL pointer");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(idx_dev)) & 3u)
        return set_err(QG_ERR_ARG, "argmax_f32: x and idx_dev must be 4-byte aligned");
    if (n <= 0) return set_err(QG_ERR_EMPTY, "argmax_f32: n=%d", n);
    argmax_f32_kernel<<<1, 1024, 0, reinterpret_cast<cudaStream_t>(stream)>>>(x, n, idx_dev);
    QG_CUDA(cudaGetLastError());
    return QG_OK;
}

int qg_device_status(void) {
    unsigned* p = block_err_ptr();
    if (!p) return set_err(QG_ERR_CUDA, "device_status: no device error word");
    unsigned v = 0;
    QG_CUDA(cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost));
    if (v) {
        const unsigned zero = 0;
        QG_CUDA(cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice));
        return set_err(QG_ERR_TIMEOUT, "a building-block kernel gave up on a bounded wait (flags 0x%x)", v);
    }
    return QG_OK;
}

}  // extern "C"
