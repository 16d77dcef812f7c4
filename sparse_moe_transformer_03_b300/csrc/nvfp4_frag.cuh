// nvfp4_frag.cuh -- NVFP4 (E2M1 codes, E4M3 block scales) weights turned into
// tensor-core A fragments in registers, shared by the NVFP4 decode kernels.
//
// NVFP4 run as W4A16 (RecursiveSI/flint vLLM recipe page, "Overview").  A
// weight is e2m1(q) * e4m3(s_block) * s_tensor with one E4M3 scale per 16
// consecutive columns of a row: one k-step of mma.sync m16n8k16.  The owned
// layout (decode_nvfp4.cu) keeps, per K block, each lane's four code bytes of
// the A fragment together and the two scales of its rows (g, g + 8) side by side.
#pragma once

#include <cuda_fp16.h>

#include "flint_common.cuh"

namespace flint {

// A fragment (f16) of one 16 x 16 block: codes = this lane's 4 code bytes,
// sc2 = E4M3 scales of its rows (g, g + 8).
__device__ __forceinline__ void nv_a_frag(uint32_t codes, uint16_t sc2, uint32_t (&a)[4]) {
    uint32_t s;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s) : "h"(sc2));
    const __half2 s2 = *reinterpret_cast<const __half2*>(&s);
    const __half2 sg = __low2half2(s2), s8 = __high2half2(s2);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint32_t h;
        asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n" : "=r"(h) : "r"(codes >> (8 * k)));
        const __half2 q = *reinterpret_cast<const __half2*>(&h);
        const __half2 r = __hmul2(q, (k & 1) ? s8 : sg);
        a[k] = *reinterpret_cast<const uint32_t*>(&r);
    }
}

__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t v) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
    const __nv_bfloat162 b = __float22bfloat162_rn(f);   // exact: at most 6 significant bits
    return *reinterpret_cast<const uint32_t*>(&b);
}

}  // namespace flint
