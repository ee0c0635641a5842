// memq_gemv_q8_0.cu -- Q8_0 GEMV and its fused decode step.
// Operation: gemv_e4m3_bench.rs (memra-engine 0.125.0), module doc, "THE COMPARISON", arm Q8_0
// (ggml block_q8_0, `synth_q8_0`).
#include "memq_gemv_kernels.cuh"

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

// Internal: this translation unit's device fault word (not part of the public header).
int memq_internal_fault_q8_0(unsigned int *out, bool clear) {
    return memq::read_fault(out, clear) == cudaSuccess ? 0 : 1;
}
