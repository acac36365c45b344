// ssm_tmap.h -- host-side construction of the TMA tensor maps the kernels
// read their [batch][L][dim] tiles through (cuTensorMapEncodeTiled, looked up
// from the driver at run time so that the library links only the runtime).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssm_internal.h"

namespace ssm {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiled encode_fn() {
    static EncodeTiled fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiled>(nullptr);
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

// [batch][L][dim] tensor, box of `box_channels` channels x `box_rows` tokens x
// 1 batch row (elements before the sequence start, past its end or past the
// last channel read as zero).
template <typename T>
inline cudaError_t make_tmap(CUtensorMap* tm, const void* base, int64_t batch, int64_t L, int64_t dim,
                      int box_channels, int box_rows = kScanStageTokens) {
    EncodeTiled fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t es = sizeof(T);
    const cuuint64_t gdim[3] = {cuuint64_t(dim), cuuint64_t(L), cuuint64_t(batch)};
    const cuuint64_t gstride[2] = {cuuint64_t(dim) * es, cuuint64_t(L) * cuuint64_t(dim) * es};
    const cuuint32_t box[3] = {cuuint32_t(box_channels), cuuint32_t(box_rows), 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    const CUresult r = fn(tm, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          3, const_cast<void*>(base), gdim, gstride, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// make_tmap with a small per-thread cache: an encoding depends only on the
// address, sizes, box and element type, so a hit is always the right map.
// Encoding costs microseconds of host time per call, which bounds short
// kernels launched back to back; callers cycle through few buffers.
template <typename T>
inline cudaError_t make_tmap_cached(CUtensorMap* tm, const void* base, int64_t batch, int64_t L,
                                    int64_t dim, int box_channels, int box_rows = kScanStageTokens) {
    struct Key {
        const void* base;
        int64_t batch, L, dim;
        int box_channels, box_rows, es;
    };
    constexpr int kEntries = 32;
    thread_local Key keys[kEntries];
    thread_local CUtensorMap maps[kEntries];
    thread_local int used = 0, next = 0;
    const Key k{base, batch, L, dim, box_channels, box_rows, int(sizeof(T))};
    for (int i = 0; i < used; ++i) {
        const Key& e = keys[i];
        if (e.base == k.base && e.batch == k.batch && e.L == k.L && e.dim == k.dim &&
            e.box_channels == k.box_channels && e.box_rows == k.box_rows && e.es == k.es) {
            *tm = maps[i];
            return cudaSuccess;
        }
    }
    const cudaError_t err = make_tmap<T>(tm, base, batch, L, dim, box_channels, box_rows);
    if (err != cudaSuccess) return err;
    keys[next] = k;
    maps[next] = *tm;
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
    return cudaSuccess;
}

// Multiprocessor count of the current device (looked up once per device).
inline int device_sms() {
    static int sms[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
    if (sms[dev] == 0) {
        int n = 0;
        sms[dev] = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
                           n > 0
                       ? n
                       : 148;
    }
    return sms[dev];
}

}  // namespace ssm
