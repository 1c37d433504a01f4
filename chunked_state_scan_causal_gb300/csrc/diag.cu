// Diagnostic: one 128x128x128 bf16 product on the tensor cores through the
// exact staging the attention kernels use (TMA into SW128 tiles, K-major and
// MN-major descriptors, TMEM accumulator, tcgen05.ld epilogue), so that every
// operand encoding can be checked against a plain matrix product.
#include "internal.h"
#include "ptx.cuh"

namespace linattn {
namespace {

__global__ void __launch_bounds__(128) diag_mma_kernel(const __grid_constant__ CUtensorMap mapA,
                                                       const __grid_constant__ CUtensorMap mapB,
                                                       int mode, float *D) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *tA = smem;
  uint8_t *tB = smem + kTileBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 2 * kTileBytes);  // [0] load, [1] mma, [2] A staged
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 4);
  __shared__ int abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 128);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmemA = tmem + 128;  // A staged in TMEM (mode 4): 64 columns of bf16 pairs

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bars[0], 2 * kTileBytes);
    tma_load_4d(&mapA, &bars[0], tA, 0, 0, 0, 0, kPolicyEvictNormal);
    tma_load_4d(&mapA, &bars[0], tA + kTileHalfBytes, 64, 0, 0, 0, kPolicyEvictNormal);
    tma_load_4d(&mapB, &bars[0], tB, 0, 0, 0, 0, kPolicyEvictNormal);
    tma_load_4d(&mapB, &bars[0], tB + kTileHalfBytes, 64, 0, 0, 0, kPolicyEvictNormal);
  }
  bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[0], 0, &abort_flag, nullptr));

  if (mode == 4 && ok) {
    // stage A (row-major, row = thread) into TMEM as packed bf16 pairs
    const uint32_t row = threadIdx.x;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int c = 0; c < 4; ++c) {  // 4 x 16 columns = 128 bf16
      uint32_t r[16];
      for (int q = 0; q < 4; ++q) {
        const uint32_t chunk = c * 4 + q;
        ld_shared_v4(smem_u32(tA) + sw128_offset(row, chunk), r[4 * q], r[4 * q + 1], r[4 * q + 2],
                     r[4 * q + 3]);
      }
      tmem_st16(tmemA + lane_base + c * 16, r);
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&bars[2]);
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[2], 0, &abort_flag, nullptr));
  }

  if (threadIdx.x == 0 && ok) {
    tc_fence_after();
    const uint32_t a = smem_u32(tA), b = smem_u32(tB);
    for (uint32_t ks = 0; ks < 8; ++ks) {
      switch (mode) {
        case 0:  // D = A B^T : A K-major, B K-major
          mma_ss(tmem, desc_kmajor(a, ks), desc_kmajor(b, ks), idesc_bf16(128, 128, false, false), ks > 0);
          break;
        case 1:  // D = A^T B : both MN-major
          mma_ss(tmem, desc_mnmajor(a, ks), desc_mnmajor(b, ks), idesc_bf16(128, 128, true, true), ks > 0);
          break;
        case 2:  // D = A B : A K-major, B MN-major
          mma_ss(tmem, desc_kmajor(a, ks), desc_mnmajor(b, ks), idesc_bf16(128, 128, false, true), ks > 0);
          break;
        case 3:  // D = A^T B^T : A MN-major, B K-major
          mma_ss(tmem, desc_mnmajor(a, ks), desc_kmajor(b, ks), idesc_bf16(128, 128, true, false), ks > 0);
          break;
        default:  // D = A B with A from TMEM
          mma_ts(tmem, tmemA + ks * 8, desc_mnmajor(b, ks), idesc_bf16(128, 128, false, true), ks > 0);
          break;
      }
    }
    mma_commit(&bars[1]);
  }
  ok = __all_sync(0xffffffffu, ok && mbar_wait(&bars[1], 0, &abort_flag, nullptr));
  tc_fence_after();
  if (ok) {
    const uint32_t row = warp * 32 + lane;
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, r);
      tmem_ld_wait();
      for (int j = 0; j < 32; ++j) D[row * 128 + c * 32 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

cudaError_t diag_mma(int mode, const void *A, const void *B, float *D, cudaStream_t s) {
  alignas(64) CUtensorMap mA, mB;
  const uint64_t dims[4] = {128, 128, 1, 1};
  const uint64_t strides[3] = {256, 256 * 128, 256 * 128};
  if (!make_tmap_bf16(&mA, A, dims, strides) || !make_tmap_bf16(&mB, B, dims, strides))
    return cudaErrorInvalidValue;
  const size_t sm = 2 * kTileBytes + 1024 + 64;
  cudaError_t e = cudaFuncSetAttribute(diag_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  TimedLaunch t(K_DIAG, s);
  diag_mma_kernel<<<1, 128, sm, s>>>(mA, mB, mode, D);
  return cudaGetLastError();
}

}  // namespace linattn
