// memq_abi.cu -- library-wide entry points: status strings, version, device fault word.
#include <cstdint>
#include <cuda_runtime.h>

#include "memq.h"

int memq_internal_fault_e4m3(unsigned int *out, bool clear);
int memq_internal_fault_blk128(unsigned int *out, bool clear);
int memq_internal_fault_q8_0(unsigned int *out, bool clear);
int memq_internal_fault_mla(unsigned int *out, bool clear);
int memq_internal_step_host_e4m3(const float *x_host, float *x_dev, const float *wn, float eps,
                                 const void *w, const float *aux, int8_t *qs, float *d, float *z,
                                 float *y_dev, float *y_host, int64_t out_f, int64_t in_f, int m,
                                 void *stream);
int memq_internal_step_host_blk128(const float *x_host, float *x_dev, const float *wn, float eps,
                                   const void *w, const float *aux, int8_t *qs, float *d, float *z,
                                   float *y_dev, float *y_host, int64_t out_f, int64_t in_f, int m,
                                   void *stream);
int memq_internal_step_host_q8_0(const float *x_host, float *x_dev, const float *wn, float eps,
                                 const void *w, const float *aux, int8_t *qs, float *d, float *z,
                                 float *y_dev, float *y_host, int64_t out_f, int64_t in_f, int m,
                                 void *stream);

extern "C" int memq_decode_step_host(int container, const float *x_host, float *x_dev,
                                     const float *wn, float eps, const void *w, const float *aux,
                                     int8_t *qs, float *d, float *z, float *y_dev, float *y_host,
                                     int64_t out_f, int64_t in_f, int m, void *stream) {
    switch (container) {
        case MEMQ_CONTAINER_E4M3:
            return memq_internal_step_host_e4m3(x_host, x_dev, wn, eps, w, aux, qs, d, z, y_dev,
                                                y_host, out_f, in_f, m, stream);
        case MEMQ_CONTAINER_E4M3_BLK128:
            return memq_internal_step_host_blk128(x_host, x_dev, wn, eps, w, aux, qs, d, z, y_dev,
                                                  y_host, out_f, in_f, m, stream);
        case MEMQ_CONTAINER_Q8_0:
            return memq_internal_step_host_q8_0(x_host, x_dev, wn, eps, w, aux, qs, d, z, y_dev,
                                                y_host, out_f, in_f, m, stream);
        default:
            return MEMQ_ERR_SHAPE;
    }
}

extern "C" int memq_device_fault(void *stream, uint32_t *fault_out) {
    if (!fault_out) return MEMQ_ERR_NULL;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MEMQ_ERR_DEVICE;
    unsigned int a = 0, b = 0, c = 0, e = 0;
    if (memq_internal_fault_e4m3(&a, true) || memq_internal_fault_blk128(&b, true) ||
        memq_internal_fault_q8_0(&c, true) || memq_internal_fault_mla(&e, true))
        return MEMQ_ERR_DEVICE;
    *fault_out = a | b | c | e;
    return MEMQ_OK;
}

extern "C" const char *memq_status_string(int status) {
    switch (status) {
        case MEMQ_OK: return "ok";
        case MEMQ_ERR_NULL: return "a required pointer is NULL";
        case MEMQ_ERR_SHAPE: return "a size is out of range or not a multiple of 32";
        case MEMQ_ERR_ALIGN: return "a pointer breaks its documented alignment";
        case MEMQ_ERR_M_RANGE: return "m is outside [1, 8]";
        case MEMQ_ERR_LAUNCH: return "the CUDA launch failed";
        case MEMQ_ERR_DEVICE: return "the device fault word could not be read";
        default: return "unknown memq status";
    }
}

extern "C" int memq_version(void) { return (1 << 16) | 1; }
