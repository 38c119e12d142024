// qsa_peaks.cu -- roofline denominators that no vendor library measures,
// built as libqsa_peaks.so beside libqsa.so and timed by the benchmark on the
// GPU it reports (CUDA events on the caller's stream):
//
//   qsa_peaks_l2_read  L2 -> SM read bandwidth.  Every thread issues 16-byte
//       loads that bypass L1 (ld.global.cg, the path the attention's cp.async.cg
//       gathers take), eight in flight, over a power-of-two buffer small enough
//       to stay resident in L2 (32 MB of the 129 MB), re-read `passes` times.
//       A warp instruction reads 512 contiguous bytes.  Bytes per launch:
//       passes * bytes.  The buffer's lines are spread over both L2 halves of
//       the two-die part, as the attention's K/V rows are.
//   qsa_peaks_l2_cpasync  the same L2 -> SM bandwidth through cp.async.cg
//       16-byte copies into shared memory (the attention kernels' path): every
//       thread keeps 8 copies in flight into a 64 KB ring of its CTA, three
//       CTAs per SM.  Bytes per launch: passes * bytes.
//   qsa_peaks_ffma     CUDA-core fp32 FMA rate: 16 independent FMA chains per
//       thread, `iters` steps each, so issue, not latency, is the limit.
//       FMAs per launch: grid * 256 * 16 * iters.
//
// These kernels are measurement only; no entry point of libqsa.so uses them.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace {

__global__ void __launch_bounds__(512) l2_read_kernel(const uint4* __restrict__ buf, size_t mask, size_t total,
                                                      unsigned* sink) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  unsigned x = 0u;
  for (; e + 7 * stride < total; e += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcg(buf + ((e + u * stride) & mask));
#pragma unroll
    for (int u = 0; u < 8; ++u) x ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; e < total; e += stride) {
    const uint4 v = __ldcg(buf + (e & mask));
    x ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (x == 0x9e3779b9u) sink[0] = x;  // keeps the loads; practically never stores
}

__global__ void __launch_bounds__(512) l2_cpasync_kernel(const uint4* __restrict__ buf, size_t mask, size_t total,
                                                          unsigned* sink) {
  extern __shared__ __align__(16) uint4 ring[];  // 512 threads x 8 chunks x 16 B = 64 KB
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(ring + threadIdx.x));
  for (; e + 7 * stride < total; e += 8 * stride) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(base + u * 512 * 16),
                   "l"(buf + ((e + u * stride) & mask))
                   : "memory");
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    asm volatile("cp.async.wait_group 1;\n" ::: "memory");  // one group of 8 copies stays in flight
  }
  for (int u = 0; e < total; e += stride, ++u)  // the last partial round: every counted byte is read
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(base + (u & 7) * 512 * 16), "l"(buf + (e & mask))
                 : "memory");
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  if (ring[threadIdx.x].x == 0x9e3779b9u && ring[threadIdx.x].y == 0x9e3779b9u) sink[0] = 1u;  // keeps the copies
}

__global__ void __launch_bounds__(256) ffma_kernel(float* out, int iters, float seed) {
  float a[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) a[j] = seed + static_cast<float>(threadIdx.x + j);
  const float m = 0.999f, c = 1e-3f;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 16; ++j) a[j] = fmaf(a[j], m, c);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) s += a[j];
  if (s == -1.f) out[0] = s;  // keeps the chains; never true for these inputs
}

}  // namespace

extern "C" {

// Reads `bytes` (a power of two, multiple of 16, at most 1 GiB) at `buf`
// `passes` times with `grid` CTAs of 512 threads.  Returns 0 or a cudaError_t.
__attribute__((visibility("default"))) int qsa_peaks_l2_read(const void* buf, size_t bytes, int passes,
                                                             unsigned* sink, int grid, void* stream) {
  if (!buf || !sink || bytes < 16 || (bytes & (bytes - 1)) || passes < 1 || grid < 1) return cudaErrorInvalidValue;
  const size_t n16 = bytes / 16;
  l2_read_kernel<<<grid, 512, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint4*>(buf), n16 - 1,
                                                                      n16 * static_cast<size_t>(passes), sink);
  return static_cast<int>(cudaGetLastError());
}

// The same read through cp.async.cg into shared memory, `grid` CTAs of 512 threads (64 KB each).
__attribute__((visibility("default"))) int qsa_peaks_l2_cpasync(const void* buf, size_t bytes, int passes,
                                                                unsigned* sink, int grid, void* stream) {
  if (!buf || !sink || bytes < 16 || (bytes & (bytes - 1)) || passes < 1 || grid < 1) return cudaErrorInvalidValue;
  constexpr int kSmem = 512 * 8 * 16;
  static const cudaError_t attr =
      cudaFuncSetAttribute(l2_cpasync_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (attr != cudaSuccess) return static_cast<int>(attr);
  const size_t n16 = bytes / 16;
  l2_cpasync_kernel<<<grid, 512, kSmem, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(buf), n16 - 1, n16 * static_cast<size_t>(passes), sink);
  return static_cast<int>(cudaGetLastError());
}

// grid CTAs of 256 threads, each thread 16 * iters FMAs.
__attribute__((visibility("default"))) int qsa_peaks_ffma(float* out, int iters, int grid, void* stream) {
  if (!out || iters < 1 || grid < 1) return cudaErrorInvalidValue;
  ffma_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(out, iters, 1.0f);
  return static_cast<int>(cudaGetLastError());
}

}  // extern "C"
