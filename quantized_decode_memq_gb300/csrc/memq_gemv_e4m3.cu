// memq_gemv_e4m3.cu -- per-tensor-scale E4M3 GEMV and its fused decode step.
// Operation: gemv_e4m3_bench.rs (memra-engine 0.125.0), module doc, "THE COMPARISON", arm E4M3.
#include "memq_gemv_kernels.cuh"

extern "C" int memq_gemv_e4m3(const uint8_t *w, const float *w_scale, const int8_t *qs,
                              const float *d, float *y, int64_t out_f, int64_t in_f, int m,
                              void *stream) {
    return memq::gemv_entry<memq::kE4M3>(w, w_scale, qs, d, y, out_f, in_f, m, stream);
}

extern "C" int memq_rmsnorm_q8_1_gemv_e4m3(const float *x, const float *wn, float eps,
                                           const uint8_t *w, const float *w_scale, int8_t *qs,
                                           float *d, float *z, float *y, int64_t out_f,
                                           int64_t in_f, int m, void *stream) {
    return memq::fused_entry<memq::kE4M3>(x, wn, eps, w, w_scale, qs, d, z, y, out_f, in_f, m,
                                          stream);
}

extern "C" int memq_gemv_e4m3_group(int count, const uint8_t *const *w,
                                    const float *const *w_scale, float *const *y,
                                    const int64_t *out_f, const int8_t *qs, const float *d,
                                    int64_t in_f, int m, void *stream) {
    return memq::group_entry<memq::kE4M3>(count, w, w_scale, y, out_f, qs, d, in_f, m, stream);
}

// Internal: this translation unit's device fault word (not part of the public header).
int memq_internal_fault_e4m3(unsigned int *out, bool clear) {
    return memq::read_fault(out, clear) == cudaSuccess ? 0 : 1;
}
