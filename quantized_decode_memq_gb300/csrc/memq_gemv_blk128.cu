// memq_gemv_blk128.cu -- block-128 scale-grid E4M3 GEMV and its fused decode step.
// Operation: gemv_e4m3_bench.rs (memra-engine 0.125.0), module doc, "THE BLOCK-128 ARM".
#include "memq_gemv_kernels.cuh"

extern "C" int memq_gemv_e4m3_blk128(const uint8_t *w, const float *grid, const int8_t *qs,
                                     const float *d, float *y, int64_t out_f, int64_t in_f, int m,
                                     void *stream) {
    return memq::gemv_entry<memq::kBlk>(w, grid, qs, d, y, out_f, in_f, m, stream);
}

extern "C" int memq_rmsnorm_q8_1_gemv_e4m3_blk128(const float *x, const float *wn, float eps,
                                                  const uint8_t *w, const float *grid, int8_t *qs,
                                                  float *d, float *z, float *y, int64_t out_f,
                                                  int64_t in_f, int m, void *stream) {
    return memq::fused_entry<memq::kBlk>(x, wn, eps, w, grid, qs, d, z, y, out_f, in_f, m,
                                         stream);
}

extern "C" int memq_gemv_e4m3_blk128_group(int count, const uint8_t *const *w,
                                           const float *const *grid, float *const *y,
                                           const int64_t *out_f, const int8_t *qs, const float *d,
                                           int64_t in_f, int m, void *stream) {
    return memq::group_entry<memq::kBlk>(count, w, grid, y, out_f, qs, d, in_f, m, stream);
}

// Internal: memq_decode_step_host for this container (the public entry point dispatches here).
int memq_internal_step_host_blk128(const float *x_host, float *x_dev, const float *wn, float eps,
                                   const void *w, const float *aux, int8_t *qs, float *d, float *z,
                                   float *y_dev, float *y_host, int64_t out_f, int64_t in_f, int m,
                                   void *stream) {
    const uint8_t *w8 = static_cast<const uint8_t *>(w);
    // the single fused launch: measured faster here than the producer + GEMV pair (C2,
    // Q8_0 4096 x 4096: 34 against 40 us per call with the copies and the wait)
    const auto step = [&]() {
        return memq_rmsnorm_q8_1_gemv_e4m3_blk128(x_dev, wn, eps, w8, aux, qs, d, z, y_dev, out_f, in_f, m, stream);
    };
    return memq::host_step_entry<memq::kBlk>(
        x_host, x_dev, wn, eps, w8, aux, qs, d, z, y_dev, y_host, out_f, in_f, m, stream, step);
}

// Internal: this translation unit's device fault word (not part of the public header).
int memq_internal_fault_blk128(unsigned int *out, bool clear) {
    return memq::read_fault(out, clear) == cudaSuccess ? 0 : 1;
}
