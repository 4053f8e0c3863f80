// Host-side helpers: the thread-local error message behind qg_last_error(),
// CUDA status mapping, and the GEMV launcher (geometry, shared memory size,
// programmatic-dependent-launch attribute).
#pragma once
#include <cstdarg>
#include <cstdio>
#include <cuda_runtime.h>

#include "../../include/qg.h"
#include "qg_gemv.cuh"

namespace qg {

int set_err(int code, const char* fmt, ...);
int cuda_err(cudaError_t e, const char* what);
int device_sms();
// Raise `kern`'s dynamic shared-memory limit to at least `smem` bytes (and
// prefer the largest carveout) on the current device, once per (kernel,
// device) and size: the attribute is per device, so a kernel configured on
// one device is configured again on the next.  Thread-safe.
int grant_smem(const void* kern, int smem);

#define QG_CUDA(call)                                              \
    do {                                                           \
        cudaError_t e_ = (call);                                   \
        if (e_ != cudaSuccess) return ::qg::cuda_err(e_, #call);   \
    } while (0)

constexpr int kCtaSmemBytes = 110 * 1024;  // per CTA: two CTAs per SM fit in 228 KB
constexpr int kStageTargetBytes = 27 * 1024;  // bulk copies of 13-27 KB stream at full rate

// Geometry for n rows of k weights (dual: two matrices streamed together)
// over at most max_ctas CTAs (0: two per SM), stages of at most max_pp row
// passes.  K is cut into slices of 32 chunks, then the binary digits of the
// remainder (16, 8, 4 chunks).
inline GemvShape gemv_geometry(int qt, bool dual, const void* w0, const void* w1, int n, int k, int pro_floats,
                               int max_ctas, unsigned* err, int* grid_out, int max_pp = 0) {
    GemvShape sh{};
    sh.w0 = static_cast<const uint8_t*>(w0);
    sh.w1 = static_cast<const uint8_t*>(w1);
    sh.n = n;
    sh.n8 = (n + 7) & ~7;
    sh.k = k;
    sh.nb = k / 256;
    sh.cr = k / 64;
    sh.err = err;
    sh.pro_floats = pro_floats;
    int c = 0;
    sh.nsl = 0;
    while (sh.cr - c >= 32 && sh.nsl < kMaxSlices) {
        sh.sl_c0[sh.nsl] = c;
        sh.sl_lg[sh.nsl++] = 5;
        c += 32;
    }
    for (int lg = 4; lg >= 2; --lg)
        if ((((sh.cr - c) >> lg) & 1) && sh.nsl < kMaxSlices) {
            sh.sl_c0[sh.nsl] = c;
            sh.sl_lg[sh.nsl++] = lg;
            c += 1 << lg;
        }
    sh.units = (n + 7) / 8;
    int grid = max_ctas > 0 ? max_ctas : 2 * device_sms();
    if (grid > sh.units) grid = sh.units;
    if (grid < 1) grid = 1;
    sh.rows_cta = 8 * ((sh.units + grid - 1) / grid);
    const int fixed = off_ring(qt, k, pro_floats, (dual ? 2 : 1) * sh.rows_cta);
    int pp = kStageTargetBytes / stage_bytes_of(qt);
    if (max_pp > 0 && pp > max_pp) pp = max_pp;
    if (pp < 1) pp = 1;
    while (pp > 1 && (kCtaSmemBytes - fixed) / (pp * stage_bytes_of(qt)) < 3) --pp;  // keep three stages in flight
    sh.pp = pp;
    int stages = (kCtaSmemBytes - fixed) / (pp * stage_bytes_of(qt));
    if (stages > kMaxStages) stages = kMaxStages;
    sh.stages = stages < 1 ? 1 : stages;
    *grid_out = grid;
    return sh;
}

// k the engine serves: a multiple of 256 whose slices fit kMaxSlices.
inline bool gemv_k_served(int k) { return k > 0 && k % 256 == 0 && k <= 16384; }

// Bytes of dynamic shared memory one GEMV launch needs.
inline int gemv_smem(const GemvShape& sh, int qt, bool dual) {
    return off_ring(qt, sh.k, sh.pro_floats, (dual ? 2 : 1) * sh.rows_cta) + sh.stages * sh.pp * stage_bytes_of(qt);
}

namespace {  // per translation unit, like the kernels they launch and configure

// Launch one GEMV-engine kernel on `st` (with programmatic stream
// serialisation when `pdl`, so the weights of this launch stream in while the
// previous kernel on the stream finishes).  err: the device error word, which
// the kernel also reads as its abort flag.
template <int QT, bool DUAL, int LAYOUT = LAYOUT_GROUPED, class Pro, class Epi>
int launch_gemv(const void* w0, const void* w1, int n, int k, const Pro& pro, const Epi& epi, cudaStream_t st,
                bool pdl, unsigned* err, const L2Prefetch& next = L2Prefetch{}, int max_ctas = 0) {
    if (!err) return set_err(QG_ERR_CUDA, "gemv: no device error word");
    int grid = 1;
    GemvShape sh = gemv_geometry(QT, DUAL, w0, w1, n, k, pro.floats(k), max_ctas, err, &grid);
    sh.next = next;
    const int smem = gemv_smem(sh, QT, DUAL);
    if (smem > 227 * 1024)
        return set_err(QG_ERR_SHAPE, "gemv: %d x %d needs %d bytes of shared memory per CTA", n, k, smem);
    auto kern = gemv_kernel<QT, LAYOUT, DUAL, Pro, Epi>;
    if (int rc = grant_smem(reinterpret_cast<const void*>(kern), smem)) return rc;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    QG_CUDA(cudaLaunchKernelEx(&cfg, kern, sh, pro, epi));
    return QG_OK;
}

// Number of K slices of a k-wide GEMV (32-chunk slices, then 16, 8, 4).
inline int gemv_slices(int k) {
    const int cr = k / 64;
    return cr / 32 + ((cr >> 4) & 1) + ((cr >> 3) & 1) + ((cr >> 2) & 1);
}

// Split-K launch (gemv_split_kernel): the slice sums of y = W x go to
// part[slice][row] (nsl * n8 floats of device scratch); the reader of y adds
// them in slice order.  W in the grouped layout.
template <int QT, class Pro>
int launch_gemv_split(const void* w0, int n, int k, const Pro& pro, cudaStream_t st, bool pdl, unsigned* err,
                      float* part, const L2Prefetch& next = L2Prefetch{}) {
    if (!err || !part) return set_err(QG_ERR_CUDA, "gemv_split: missing scratch");
    // the kernel splits its tasks with 32-bit products (blockIdx + 1) * tasks
    if (n <= 0 || n > (1 << 20)) return set_err(QG_ERR_SHAPE, "gemv_split: n must be in [1, 2^20]");
    int grid = 1;
    GemvShape sh = gemv_geometry(QT, false, w0, nullptr, n, k, pro.floats(k), 0, err, &grid);
    const long long tasks = static_cast<long long>(sh.units) * sh.nsl;
    grid = static_cast<int>(tasks < 2LL * device_sms() ? tasks : 2LL * device_sms());
    sh.rows_cta = 0;
    const int fixed = off_ring(QT, k, sh.pro_floats, 0);
    int stages = (kCtaSmemBytes - fixed) / (sh.pp * stage_bytes_of(QT));
    sh.stages = stages < 1 ? 1 : (stages > kMaxStages ? kMaxStages : stages);
    sh.part = part;
    sh.next = next;
    const int smem = fixed + sh.stages * sh.pp * stage_bytes_of(QT);
    auto kern = gemv_split_kernel<QT, Pro>;
    if (int rc = grant_smem(reinterpret_cast<const void*>(kern), smem)) return rc;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    QG_CUDA(cudaLaunchKernelEx(&cfg, kern, sh, pro));
    return QG_OK;
}

}  // namespace

// Plain launch of a non-engine kernel with the PDL attribute.
template <class... KArgs, class... Args>
int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
               Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    QG_CUDA(cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...));
    return QG_OK;
}

}  // namespace qg
