/*
 * Example operator module, compiled on its own to a relocatable sm_103a cubin
 * (nvcc -cubin -rdc=true) and handed to gpuos_load_module / gpuos_register_op
 * ("GPUOS: A GPU Operating System Primitive for Transparent Operation
 * Fusion", §3 Q2 "3. Dynamic Operator Table": load the operator through the
 * driver API, resolve its symbol to a device-function pointer, write it into
 * the inactive table slot, flip the version).
 *
 * The library links this object with its relocatable executor build before
 * the executor's launch, so the functions live in the executor's own module
 * (a device-function pointer is only callable inside the module that holds
 * its code). Each op is exported as a __device__ variable holding the
 * function's address, read after linking with cuModuleGetGlobal. The
 * functions follow the executor's op signature and stay within its register
 * budget (the build caps them at the executor's register count).
 *
 *   gpuos_ext_sub   out = a - b, element-wise fp32/bf16, same tiling as the
 *                   built-in add (it can replace op 1 in a hot swap)
 *   gpuos_ext_scale out = a * fparam[0], fp32, user op: tile t covers
 *                   elements [1024 t, 1024 t + 1024), the caller sets ntiles
 */
#include <cuda_bf16.h>
#include <stdint.h>

#include "gpuos_internal.h"

static __device__ __forceinline__ float bf1(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
static __device__ __forceinline__ uint16_t to_bf(float x)
{
    __nv_bfloat16 v = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&v);
}

extern "C" __device__ __noinline__ int gpuos_ext_sub(const gpuos_devdesc *d, uint32_t tile)
{
    const uint32_t lane = threadIdx.x & 31u;
    const bool bf = d->dtype == GPUOS_BF16;
    const uint64_t n = d->dims[0];
    /* the built-in element-wise ops' tile rule: ntiles ranges of
     * round_up(ceil(n / ntiles), GPUOS_EW_ALIGN) elements (so the op can
     * stand in for add, whose ntiles the library computes) */
    const uint64_t nt = d->ntiles ? d->ntiles : 1u;
    const uint64_t T = ((n + nt - 1) / nt + GPUOS_EW_ALIGN - 1) / GPUOS_EW_ALIGN * GPUOS_EW_ALIGN;
    const uint64_t start = (uint64_t)tile * T;
    if (start >= n) return GPUOS_ST_OK;
    const uint64_t end = (n - start) < T ? n : start + T;
    if (bf) {
        const uint16_t *a = reinterpret_cast<const uint16_t *>(d->a);
        const uint16_t *b = reinterpret_cast<const uint16_t *>(d->b);
        uint16_t *o = reinterpret_cast<uint16_t *>(d->out);
        for (uint64_t i = start + lane; i < end; i += 32) o[i] = to_bf(__fsub_rn(bf1(__ldcg(a + i)), bf1(__ldcg(b + i))));
    } else {
        const float *a = reinterpret_cast<const float *>(d->a);
        const float *b = reinterpret_cast<const float *>(d->b);
        float *o = reinterpret_cast<float *>(d->out);
        for (uint64_t i = start + lane; i < end; i += 32) o[i] = __fsub_rn(__ldcg(a + i), __ldcg(b + i));
    }
    return GPUOS_ST_OK;
}

extern "C" __device__ __noinline__ int gpuos_ext_scale(const gpuos_devdesc *d, uint32_t tile)
{
    const uint32_t lane = threadIdx.x & 31u;
    if (d->dtype != GPUOS_F32) return GPUOS_ST_BAD_ARGS;
    const uint64_t n = d->dims[0];
    const uint64_t start = (uint64_t)tile * 1024;
    const float s = d->fparam[0];
    const float *a = reinterpret_cast<const float *>(d->a);
    float *o = reinterpret_cast<float *>(d->out);
    for (uint64_t i = start + lane; i < start + 1024 && i < n; i += 32) o[i] = __fmul_rn(__ldcg(a + i), s);
    return GPUOS_ST_OK;
}

extern "C" __device__ gpuos_op_fn gpuos_ext_sub_ptr = gpuos_ext_sub;
extern "C" __device__ gpuos_op_fn gpuos_ext_scale_ptr = gpuos_ext_scale;

