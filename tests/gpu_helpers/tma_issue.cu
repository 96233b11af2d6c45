// Test helper: throughput of small tiled TMA loads against the number of
// warps issuing them. Each CTA (one per SM) has W warps; per batch, lanes
// 0..ops-1 of every warp each issue one box_rows x 64 bf16 (128-byte rows,
// 128-byte swizzle) load at a pseudo-random row of a large matrix into the
// warp's own shared-memory region, lane 0 sets the batch's expected bytes on
// the warp's mbarrier, and the warp waits for them (bounded, 2 s; a timeout
// sets *err). Comparing W = 1 with 2 x ops against W = 2 with ops each, the
// same bytes are in flight: a gain means one warp's issue, not the copy
// engine, was the limit.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace {

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void tma_issue_kernel(const __grid_constant__ CUtensorMap m, int rows, int box_rows, int ops,
                                 int batches, int* err) {
  extern __shared__ uint8_t raw[];
  __shared__ __align__(8) uint64_t bar[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t box_bytes = (uint32_t)box_rows * 128u;
  const uint32_t region = (uint32_t)ops * box_bytes;
  uint8_t* base = raw + ((1024u - (smem_addr(raw) & 1023u)) & 1023u) + (size_t)warp * region;
  const uint32_t b = smem_addr(&bar[warp]);
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  const uint32_t seed = (blockIdx.x * 1315423911u) ^ (warp * 2654435761u);
  const int row_blocks = rows / box_rows;
  for (int it = 0; it < batches; ++it) {
    if (lane == 0)
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(region) : "memory");
    __syncwarp();
    if (lane < ops) {
      uint32_t h = seed ^ (uint32_t)(it * 40503 + lane * 9973);
      h ^= h >> 16;
      h *= 0x7feb352du;
      h ^= h >> 15;
      h *= 0x846ca68bu;
      h ^= h >> 16;
      const int row = (int)(h % (uint32_t)row_blocks) * box_rows;
      const int col = (int)((h >> 8) % 32u) * 64;   // one of 32 64-column halves of a 4 KB row
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
              smem_addr(base + (size_t)lane * box_bytes)),
          "l"(reinterpret_cast<uint64_t>(&m)), "r"(col), "r"(row), "r"(b)
          : "memory");
    }
    const uint64_t t0 = now_ns();
    for (;;) {
      uint32_t done;
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(done)
          : "r"(b), "r"((uint32_t)(it & 1))
          : "memory");
      if (done) break;
      if (now_ns() - t0 > 2000000000ull) {
        if (lane == 0) atomicOr(err, 1);
        return;
      }
    }
    __syncwarp();
  }
}

}  // namespace

// GB/s of box loads over `ctas` CTAs of `warps` warps, `ops` boxes per warp
// per batch; buf is a [rows, 2048] bf16 matrix. Negative on a setup error.
extern "C" double tma_issue_rate(void* buf, int rows, int box_rows, int warps, int ops, int batches, int ctas,
                                 int* err) {
  if (warps < 1 || warps > 32 || ops < 1 || ops > 32 || box_rows < 8 || box_rows > 256 || rows < box_rows) return -1.0;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      fn == nullptr)
    return -2.0;
  CUtensorMap m;
  cuuint64_t dims[2] = {2048, (cuuint64_t)rows};
  cuuint64_t strides[1] = {2048 * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  if (reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn)(
          &m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, buf, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return -3.0;
  const size_t smem = (size_t)warps * ops * box_rows * 128 + 1024;
  if (smem > 200 * 1024 ||
      cudaFuncSetAttribute(tma_issue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return -4.0;
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  tma_issue_kernel<<<ctas, 32 * warps, smem>>>(m, rows, box_rows, ops, 2, err);   // warm-up
  cudaEventRecord(a);
  tma_issue_kernel<<<ctas, 32 * warps, smem>>>(m, rows, box_rows, ops, batches, err);
  cudaEventRecord(b);
  double gbs = -5.0;
  if (cudaEventSynchronize(b) == cudaSuccess) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    gbs = (double)ctas * warps * batches * ops * box_rows * 128.0 / (ms * 1e-3) / 1e9;
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  return gbs;
}
