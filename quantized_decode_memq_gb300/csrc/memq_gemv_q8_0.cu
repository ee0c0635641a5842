// memq_gemv_q8_0.cu -- Q8_0 GEMV and its fused decode step.
// Operation: gemv_e4m3_bench.rs (memra-engine 0.125.0), module doc, "THE COMPARISON", arm Q8_0
// (ggml block_q8_0, `synth_q8_0`).
#include "memq_gemv_kernels.cuh"

namespace memq {
namespace {

// Q8_0 calls choose between two arithmetics: the tensor-core paths (the K-outer kernel and the
// tile kernel's kQ80T, bit-identical to each other) and dp4a.  The tensor cores serve a call
// when K-outer applies (q80_kouter_applies: m >= 2 on CTAs of 8 to 16 rows) or when
// q80_on_tensor_cores says so; K-outer is tried first.
inline bool q80_tensor_path(int nmat, const int64_t *out_f, int64_t rows_all, int64_t in_f, int m,
                            const int8_t *qs, const float *d, const DeviceInfo &info) {
    return q80_kouter_applies(nmat, out_f, in_f, m, qs, d, info) ||
           q80_on_tensor_cores(rows_all, in_f, m);
}

inline int q80_gemv_entry(const uint8_t *w, const int8_t *qs, const float *d, float *y,
                          int64_t out_f, int64_t in_f, int m, void *stream) {
    const int rc = check_gemv_args<kQ80>(w, nullptr, qs, d, y, out_f, in_f, m);
    if (rc >= 0) return rc;
    int dev = 0;
    DeviceInfo info;
    if (device_info(dev, info) != cudaSuccess) return MEMQ_ERR_LAUNCH;
    if (fast_path_ok<kQ80T>(w, qs, in_f) && q80_kouter_applies(1, &out_f, in_f, m, qs, d, info)) {
        const float *aux = nullptr;
        const cudaError_t ek = launch_kouter_m<kQ80T>(m, 1, &w, &aux, &y, &out_f, qs, d, in_f, dev,
                                                      info, static_cast<cudaStream_t>(stream));
        if (ek != cudaErrorNotSupported) return ek == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
        // a ring too shallow for the K-outer plan (it always fits at m = 2): the tile kernel's
        // tensor-core path
        if (m >= kQ80MmaMinM) return gemv_entry<kQ80T>(w, nullptr, qs, d, y, out_f, in_f, m, stream);
        return gemv_entry<kQ80>(w, nullptr, qs, d, y, out_f, in_f, m, stream);
    }
    if (q80_on_tensor_cores(out_f, in_f, m))
        return gemv_entry<kQ80T>(w, nullptr, qs, d, y, out_f, in_f, m, stream);
    return gemv_entry<kQ80>(w, nullptr, qs, d, y, out_f, in_f, m, stream);
}

// A Q8_0 group runs as one launch only if its path (tensor cores or dp4a) is the one each of its
// matrices takes alone, so that every output equals the single call bit for bit; otherwise it
// runs one call per matrix.
inline int q80_group_entry(int count, const uint8_t *const *w, float *const *y,
                           const int64_t *out_f, const int8_t *qs, const float *d, int64_t in_f,
                           int m, void *stream) {
    if (count < 1 || count > kMaxGroup) return MEMQ_ERR_SHAPE;
    if (!w || !y || !out_f) return MEMQ_ERR_NULL;
    int64_t rows_all = 0;
    bool fast = true;
    for (int i = 0; i < count; ++i) {
        const int rc = check_gemv_args<kQ80>(w[i], nullptr, qs, d, y[i], out_f[i], in_f, m);
        if (rc > 0) return rc;
        if (rc == MEMQ_OK) return MEMQ_ERR_SHAPE;  // an empty matrix in a group
        rows_all += out_f[i];
        fast = fast && fast_path_ok<kQ80T>(w[i], qs, in_f);
    }
    int dev = 0;
    DeviceInfo info;
    if (device_info(dev, info) != cudaSuccess) return MEMQ_ERR_LAUNCH;
    const bool tensor = q80_tensor_path(count, out_f, rows_all, in_f, m, qs, d, info);
    bool same = fast;
    for (int i = 0; i < count && same; ++i)
        same = q80_tensor_path(1, &out_f[i], out_f[i], in_f, m, qs, d, info) == tensor;
    if (same && tensor && q80_kouter_applies(count, out_f, in_f, m, qs, d, info)) {
        const float *aux[kMaxGroup] = {};
        const cudaError_t ek = launch_kouter_m<kQ80T>(m, count, w, aux, y, out_f, qs, d, in_f, dev,
                                                      info, static_cast<cudaStream_t>(stream));
        if (ek != cudaErrorNotSupported) return ek == cudaSuccess ? MEMQ_OK : MEMQ_ERR_LAUNCH;
        same = m >= kQ80MmaMinM;
    }
    if (!same) {
        for (int i = 0; i < count; ++i) {
            const int rc = q80_gemv_entry(w[i], qs, d, y[i], out_f[i], in_f, m, stream);
            if (rc != MEMQ_OK) return rc;
        }
        return MEMQ_OK;
    }
    if (tensor) return group_entry<kQ80T>(count, w, nullptr, y, out_f, qs, d, in_f, m, stream);
    return group_entry<kQ80>(count, w, nullptr, y, out_f, qs, d, in_f, m, stream);
}

}  // namespace
}  // namespace memq

extern "C" int memq_gemv_q8_0(const void *w, const int8_t *qs, const float *d, float *y,
                              int64_t out_f, int64_t in_f, int m, void *stream) {
    return memq::q80_gemv_entry(static_cast<const uint8_t *>(w), qs, d, y, out_f, in_f, m, stream);
}

extern "C" int memq_rmsnorm_q8_1_gemv_q8_0(const float *x, const float *wn, float eps,
                                           const void *w, int8_t *qs, float *d, float *z,
                                           float *y, int64_t out_f, int64_t in_f, int m,
                                           void *stream) {
    const uint8_t *w8 = static_cast<const uint8_t *>(w);
    if (memq::q80_on_tensor_cores(out_f, in_f, m))
        return memq::fused_entry<memq::kQ80T>(x, wn, eps, w8, nullptr, qs, d, z, y, out_f, in_f, m,
                                              stream);
    return memq::fused_entry<memq::kQ80>(x, wn, eps, w8, nullptr, qs, d, z, y, out_f, in_f, m,
                                         stream);
}

extern "C" int memq_gemv_q8_0_group(int count, const void *const *w, float *const *y,
                                    const int64_t *out_f, const int8_t *qs, const float *d,
                                    int64_t in_f, int m, void *stream) {
    if (count < 1 || count > memq::kMaxGroup) return MEMQ_ERR_SHAPE;
    if (!w || !out_f) return MEMQ_ERR_NULL;
    const uint8_t *w8[memq::kMaxGroup];
    for (int i = 0; i < count; ++i) w8[i] = static_cast<const uint8_t *>(w[i]);
    return memq::q80_group_entry(count, w8, y, out_f, qs, d, in_f, m, stream);
}

// Internal: memq_decode_step_host for this container (the public entry point dispatches here).
int memq_internal_step_host_q8_0(const float *x_host, float *x_dev, const float *wn, float eps,
                                 const void *w, const float *aux, int8_t *qs, float *d, float *z,
                                 float *y_dev, float *y_host, int64_t out_f, int64_t in_f, int m,
                                 void *stream) {
    const uint8_t *w8 = static_cast<const uint8_t *>(w);
    // the single fused launch: measured faster here than the producer + GEMV pair (C2,
    // Q8_0 4096 x 4096: 34 against 40 us per call with the copies and the wait)
    const auto step = [&]() {
        return memq_rmsnorm_q8_1_gemv_q8_0(x_dev, wn, eps, w, qs, d, z, y_dev, out_f, in_f, m, stream);
    };
    return memq::host_step_entry<memq::kQ80>(
        x_host, x_dev, wn, eps, w8, aux, qs, d, z, y_dev, y_host, out_f, in_f, m, stream, step);
}

// Internal: this translation unit's device fault word (not part of the public header).
int memq_internal_fault_q8_0(unsigned int *out, bool clear) {
    return memq::read_fault(out, clear) == cudaSuccess ? 0 : 1;
}
