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

#define QG_CUDA(call)                                              \
    do {                                                           \
        cudaError_t e_ = (call);                                   \
        if (e_ != cudaSuccess) return ::qg::cuda_err(e_, #call);   \
    } while (0)

// Bytes of dynamic shared memory one GEMV launch needs.
inline int gemv_smem(int qt, bool dual, int k, int pro_floats, int rows_cta, int stages, int stage_bytes) {
    return off_ring(qt, k, pro_floats, (dual ? 2 : 1) * rows_cta) + stages * stage_bytes;
}

constexpr int kStageMaxBytes = 16 * 1024;  // one stage of the ring
constexpr int kCtaSmemBytes = 110 * 1024;  // per CTA: two CTAs per SM fit in 228 KB

// Geometry for n rows of k weights (dual: two matrices streamed together).
inline GemvShape gemv_geometry(int qt, bool dual, const void* w0, const void* w1, int n, int k, int pro_floats,
                               int max_ctas, unsigned* err, int* grid_out) {
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
    const int per_row = (qt == QT_Q4K ? 144 : 210) * sh.nb * (dual ? 2 : 1);
    // lanes per row: the largest power of two <= 32 dividing the chunk count,
    // widened while one pass of 8 warps would not fit a stage
    int G = 1;
    while (G < 32 && sh.cr % (2 * G) == 0) G *= 2;
    while (G < 32 && 8 * (32 / G) * per_row > kStageMaxBytes) G *= 2;
    sh.lg = 0;
    while ((1 << sh.lg) < G) ++sh.lg;
    const int unit_rows = 8 * (32 / G);  // rows of one pass of the 8 consumer warps
    sh.units = (n + 7) / 8;
    int grid = max_ctas > 0 ? max_ctas : 2 * device_sms();
    if (grid > sh.units) grid = sh.units;
    if (grid < 1) grid = 1;
    const int rows_cta = 8 * ((sh.units + grid - 1) / grid);
    sh.rows_cta = rows_cta;
    int rs = unit_rows * (kStageMaxBytes / (unit_rows * per_row) > 0 ? kStageMaxBytes / (unit_rows * per_row) : 1);
    const int need = ((rows_cta + unit_rows - 1) / unit_rows) * unit_rows;
    if (rs > need) rs = need;
    sh.rs = rs;
    sh.stage_bytes = rs * per_row;
    int stages = (rows_cta + rs - 1) / rs;
    if (stages > kMaxStages) stages = kMaxStages;
    const int fixed = off_ring(qt, k, pro_floats, (dual ? 2 : 1) * rows_cta);
    while (stages > 1 && fixed + stages * sh.stage_bytes > kCtaSmemBytes) --stages;
    sh.stages = stages < 1 ? 1 : stages;
    *grid_out = grid;
    return sh;
}

// Launch one GEMV-engine kernel on `st` (with programmatic stream
// serialisation when `pdl`, so the weights of this launch stream in while the
// previous kernel on the stream finishes).
template <int QT, bool DUAL, class Pro, class Epi>
int launch_gemv(const void* w0, const void* w1, int n, int k, const Pro& pro, const Epi& epi, cudaStream_t st,
                bool pdl, unsigned* err, const L2Prefetch& next = L2Prefetch{}, int max_ctas = 0) {
    int grid = 1;
    GemvShape sh = gemv_geometry(QT, DUAL, w0, w1, n, k, pro.floats(k), max_ctas, err, &grid);
    sh.next = next;
    const int smem = gemv_smem(QT, DUAL, k, sh.pro_floats, sh.rows_cta, sh.stages, sh.stage_bytes);
    auto kern = gemv_kernel<QT, DUAL, Pro, Epi>;
    static int configured = 0;  // per instantiation: largest dynamic smem granted so far
    if (smem > configured) {
        QG_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        QG_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     static_cast<int>(cudaSharedmemCarveoutMaxShared)));
        configured = smem;
    }
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
