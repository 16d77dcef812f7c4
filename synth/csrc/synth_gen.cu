// synth_gen.cu -- device copy of the seeded input generator of synth/gen.py.
//
// Draws the same SplitMix64 counter streams and Box-Muller normals as the
// numpy generator, so multi-gigabyte weight stacks are produced directly in
// device memory.  Input generation only: nothing of the MoE layer's
// arithmetic is here.  SplitMix64: Steele, Lea & Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014 (the output finaliser with
// constants 0xBF58476D1CE4E5B9 / 0x94D049BB133111EB and the golden-ratio
// increment 0x9E3779B97F4A7C15).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define SYNTH_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t stream_key(uint32_t seed, uint32_t layer, uint32_t tensor) {
    return mix64((uint64_t(seed) << 32) | (uint64_t(layer & 0xFFFF) << 16) | uint64_t(tensor & 0xFFFF));
}

__device__ __forceinline__ double uniform01(uint64_t key, uint64_t i) {
    const uint64_t r = mix64(key + (i + 1) * kGolden);
    return (double(r >> 11) + 0.5) * 0x1.0p-53;
}

// normal deviates 2p and 2p+1 of the stream
__device__ __forceinline__ void normal_pair(uint64_t key, uint64_t p, double& z0, double& z1) {
    const double u1 = uniform01(key, 2 * p);
    const double u2 = uniform01(key, 2 * p + 1);
    const double rad = sqrt(-2.0 * log(u1));
    const double theta = (2.0 * 3.141592653589793) * u2;
    z0 = rad * cos(theta);
    z1 = rad * sin(theta);
}

__device__ __forceinline__ uint16_t bf16_bits_of(double v) {
    const float f = __double2float_rn(v);
    const __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<const uint16_t*>(&b);
}

// element i of dst = bf16(float(std * z_{start + i}))
__global__ void fill_normal_bf16_kernel(uint16_t* dst, uint64_t n, uint64_t start, uint64_t key, double std_) {
    const uint64_t npairs = (n + (start & 1) + 1) / 2;
    const uint64_t p0 = start / 2;
    for (uint64_t q = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; q < npairs;
         q += (uint64_t)gridDim.x * blockDim.x) {
        double z0, z1;
        normal_pair(key, p0 + q, z0, z1);
        const uint64_t e0 = 2 * (p0 + q);   // stream index of z0
        if (e0 >= start && e0 - start < n) dst[e0 - start] = bf16_bits_of(std_ * z0);
        if (e0 + 1 >= start && e0 + 1 - start < n) dst[e0 + 1 - start] = bf16_bits_of(std_ * z1);
    }
}

// n_tensors consecutive tensors of `elems` elements each; tensor i is the
// stream (seed, layer, tensor0 + i * tensor_stride)
__global__ void fill_normal_bf16_batched_kernel(uint16_t* dst, uint32_t n_tensors, uint64_t elems, uint32_t seed,
                                                uint32_t layer, uint32_t tensor0, uint32_t tensor_stride,
                                                double std_) {
    const uint64_t pairs = elems / 2;   // elems is even
    const uint64_t total = pairs * n_tensors;
    for (uint64_t q = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; q < total;
         q += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t ti = uint32_t(q / pairs);
        const uint64_t p = q - uint64_t(ti) * pairs;
        double z0, z1;
        normal_pair(stream_key(seed, layer, tensor0 + ti * tensor_stride), p, z0, z1);
        uint16_t* d = dst + uint64_t(ti) * elems + 2 * p;
        d[0] = bf16_bits_of(std_ * z0);
        d[1] = bf16_bits_of(std_ * z1);
    }
}

__global__ void fill_normal_f32_kernel(float* dst, uint64_t n, uint64_t key, double std_) {
    for (uint64_t q = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; q < (n + 1) / 2;
         q += (uint64_t)gridDim.x * blockDim.x) {
        double z0, z1;
        normal_pair(key, q, z0, z1);
        dst[2 * q] = __double2float_rn(std_ * z0);
        if (2 * q + 1 < n) dst[2 * q + 1] = __double2float_rn(std_ * z1);
    }
}

// ---------------------------------------------------------------------------
// NVFP4 encoding of bf16 matrices (the same steps, in the same fp32
// operations, as synth/gen.py nvfp4_quantize)
// ---------------------------------------------------------------------------

// max |w| of each matrix, as the bits of a non-negative float (which order
// like unsigned integers)
__global__ void amax_kernel(const uint16_t* w, uint64_t per_mat, uint32_t* amax_bits) {
    const uint32_t m = blockIdx.y;
    const uint16_t* src = w + uint64_t(m) * per_mat;
    uint32_t mx = 0;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < per_mat;
         i += (uint64_t)gridDim.x * blockDim.x)
        mx = max(mx, uint32_t(src[i] & 0x7FFFu) << 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    __shared__ uint32_t part[32];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int k = 1; k < (int)(blockDim.x >> 5); ++k) mx = max(mx, part[k]);
        atomicMax(&amax_bits[m], mx);
    }
}

// non-negative float -> E4M3 code, round to nearest even, saturating at 448
__device__ uint8_t e4m3_encode_rn_sat(float v) {
    if (!(v > 0.f)) return 0;
    int ex;
    (void)frexpf(v, &ex);                 // v = mant * 2^ex, mant in [0.5, 1)
    const int ue = ex - 1;
    const int step = ue < -6 ? -9 : ue - 3;
    const float q = rintf(ldexpf(v, -step));
    int code;
    if (ue < -6) {
        code = int(q);
    } else {
        int m = int(q) - 8, e = ue + 7;
        if (q >= 16.f) {
            e += 1;
            m = 0;
        }
        code = (e << 3) | m;
    }
    return uint8_t(min(code, 0x7E));
}

__device__ float e4m3_decode_f32(uint8_t c) {
    const int e = (c >> 3) & 15, m = c & 7;
    const float v = e == 0 ? ldexpf(float(m) / 8.f, -6) : ldexpf(1.f + float(m) / 8.f, e - 7);
    return (c & 0x80) ? -v : v;
}

// float -> E2M1 code: magnitude index into {0, .5, 1, 1.5, 2, 3, 4, 6}, round
// to nearest with ties to even, clamped at 6; bit 3 = sign (none for zero)
__device__ uint8_t e2m1_encode_rn(float v) {
    const float a = fabsf(v);
    uint8_t i = 7;
    if (a <= 5.0f) i = 6;
    if (a < 3.5f) i = 5;
    if (a <= 2.5f) i = 4;
    if (a < 1.75f) i = 3;
    if (a <= 1.25f) i = 2;
    if (a < 0.75f) i = 1;
    if (a <= 0.25f) i = 0;
    return uint8_t(i | ((v < 0.f && i > 0) ? 8 : 0));
}

// one thread per block of 16 consecutive elements of a row
__global__ void nvfp4_quant_kernel(const uint16_t* w, uint32_t n_mat, uint32_t R, uint32_t K,
                                   const uint32_t* amax_bits, uint8_t* packed, uint8_t* scales, float* tscale) {
    const uint64_t per = uint64_t(R) * (K / 16);
    for (uint64_t b = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; b < per * n_mat;
         b += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t m = uint32_t(b / per);
        const uint64_t bi = b - uint64_t(m) * per;
        const float amax = __uint_as_float(amax_bits[m]);
        const float s_t = amax == 0.f ? 1.f : __fdiv_rn(amax, 2688.0f);
        if (bi == 0) tscale[m] = s_t;
        const uint16_t* src = w + uint64_t(m) * R * K + bi * 16;
        float v[16], amax_b = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            v[k] = __uint_as_float(uint32_t(src[k]) << 16);
            amax_b = fmaxf(amax_b, fabsf(v[k]));
        }
        const float denom = __fmul_rn(6.0f, s_t);
        const uint8_t sb = e4m3_encode_rn_sat(__fdiv_rn(amax_b, denom));
        const float scale = __fmul_rn(e4m3_decode_f32(sb), s_t);
        const float safe = scale > 0.f ? scale : 1.f;
        uint8_t* pk = packed + uint64_t(m) * R * (K / 2) + bi * 8;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint8_t q0 = scale > 0.f ? e2m1_encode_rn(__fdiv_rn(v[2 * k], safe)) : 0;
            const uint8_t q1 = scale > 0.f ? e2m1_encode_rn(__fdiv_rn(v[2 * k + 1], safe)) : 0;
            pk[k] = uint8_t(q0 | (q1 << 4));
        }
        scales[uint64_t(m) * per + bi] = sb;
    }
}

int grid_for(uint64_t items) {
    uint64_t g = (items + 255) / 256;
    if (g > 148ull * 64) g = 148ull * 64;
    if (g < 1) g = 1;
    return int(g);
}

}  // namespace

// dst[i] = bf16(std * N_{start+i}) of stream (seed, layer, tensor), i < n.
SYNTH_API int synth_fill_normal_bf16(void* dst, uint64_t n, uint64_t start, uint32_t seed, uint32_t layer,
                                     uint32_t tensor, double std_, cudaStream_t s) {
    if (!dst || n == 0) return 1;
    const uint64_t npairs = (n + (start & 1) + 1) / 2;
    fill_normal_bf16_kernel<<<grid_for(npairs), 256, 0, s>>>(static_cast<uint16_t*>(dst), n, start,
                                                            stream_key(seed, layer, tensor), std_);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

// Tensor i of n_tensors (each `elems` bf16, elems even) gets stream
// (seed, layer, tensor0 + i * tensor_stride).
SYNTH_API int synth_fill_normal_bf16_batched(void* dst, uint32_t n_tensors, uint64_t elems, uint32_t seed,
                                             uint32_t layer, uint32_t tensor0, uint32_t tensor_stride, double std_,
                                             cudaStream_t s) {
    if (!dst || n_tensors == 0 || elems == 0 || (elems & 1)) return 1;
    fill_normal_bf16_batched_kernel<<<148 * 16, 256, 0, s>>>(static_cast<uint16_t*>(dst), n_tensors, elems, seed,
                                                            layer, tensor0, tensor_stride, std_);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

// dst[i] = float(std * N_i), i < n.
SYNTH_API int synth_fill_normal_f32(float* dst, uint64_t n, uint32_t seed, uint32_t layer, uint32_t tensor,
                                    double std_, cudaStream_t s) {
    if (!dst || n == 0) return 1;
    fill_normal_f32_kernel<<<grid_for((n + 1) / 2), 256, 0, s>>>(dst, n, stream_key(seed, layer, tensor), std_);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

// NVFP4 encoding of n_mat bf16 matrices [R][K] stored one after another:
// packed [n_mat][R][K/2], scales [n_mat][R][K/16], tscale [n_mat].
// amax_scratch: n_mat uint32 of device memory (overwritten).
SYNTH_API int synth_nvfp4_quantize(const void* w, uint32_t n_mat, uint32_t R, uint32_t K, void* packed,
                                   void* scales, float* tscale, uint32_t* amax_scratch, cudaStream_t s) {
    if (!w || !packed || !scales || !tscale || !amax_scratch || n_mat == 0 || R == 0 || K % 16) return 1;
    if (cudaMemsetAsync(amax_scratch, 0, n_mat * sizeof(uint32_t), s) != cudaSuccess) return 2;
    amax_kernel<<<dim3(64, n_mat), 256, 0, s>>>(static_cast<const uint16_t*>(w), uint64_t(R) * K, amax_scratch);
    const uint64_t blocks = uint64_t(n_mat) * R * (K / 16);
    nvfp4_quant_kernel<<<grid_for(blocks), 256, 0, s>>>(static_cast<const uint16_t*>(w), n_mat, R, K, amax_scratch,
                                                         static_cast<uint8_t*>(packed),
                                                         static_cast<uint8_t*>(scales), tscale);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
