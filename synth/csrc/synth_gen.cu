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
