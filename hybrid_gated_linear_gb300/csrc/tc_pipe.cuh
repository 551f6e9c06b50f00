// tc_pipe.cuh -- pieces shared by the tile kernels built on tc_sm100.cuh: the per-CTA
// barrier block with bounded waits, operand descriptors for 128-byte-swizzled tiles,
// swizzled bf16 stores, and TMA tile stores.
#pragma once

#include "tc_sm100.cuh"

namespace lz {
namespace tc {

constexpr long long kWaitCycles = 2000000000ll;  // ~1 s of SM clock per wait
constexpr uint64_t kDrainNs = 1000000000ull;     // 1 s for the exit drains

template <int NB>
struct Ctl {
  uint64_t bar[NB];
  uint32_t tmem;
  int abort;
};

// Bounded wait: gives up (and raises the CTA's abort flag) after `limit` SM clock cycles
// (kWaitCycles unless a self-test asks for less), or as soon as another role has aborted.
template <int NB>
__device__ __forceinline__ bool wait_bar(Ctl<NB>* ctl, int i, uint32_t parity,
                                         long long limit = kWaitCycles) {
  uint64_t* b = &ctl->bar[i];
  if (mbar_try_wait(b, parity)) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int k = 0; k < 32; ++k)
      if (mbar_try_wait(b, parity)) return true;
    if (*(volatile int*)&ctl->abort) return false;
    if (clock64() - t0 > limit) {
      *(volatile int*)&ctl->abort = 1;
      return false;
    }
  }
}

// Waits, with a time limit of its own, for the phase `armed` - 1 of a barrier (the last
// one armed); used only while leaving, so that no copy or MMA is left in flight.
template <int NB>
__device__ __forceinline__ void drain_bar(Ctl<NB>* ctl, int i, uint32_t armed, uint64_t t0) {
  if (armed == 0) return;
  while (!mbar_try_wait(&ctl->bar[i], (armed - 1) & 1))
    if (globaltimer_ns() - t0 > kDrainNs) break;
}

// K-major SW128 descriptor for k-step j (16 elements) of a tile of `rows` rows stored as
// 64-column blocks of rows x 128 B.
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int rows, int j) {
  return smem_desc(base + (uint32_t)((j * 16) >> 6) * (uint32_t)rows * 128u + (uint32_t)((j * 16) & 63) * 2u,
                   16, 1024, kSw128);
}

// MN-major SW128 descriptor for k-step j of a tile whose `rows` rows are the K index and
// whose 128 columns (two 64-column blocks) are the M or N index.
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int rows, int j) {
  return smem_desc(base + (uint32_t)j * 2048u, (uint32_t)rows * 128u, 1024, kSw128);
}

// 16 consecutive columns of one row of a SW128 bf16 tile.
__device__ __forceinline__ void store16_bf16(unsigned char* tile, int rows, int row, int col,
                                             const float (&v)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
  *reinterpret_cast<uint4*>(tile + sw128_offset(row, col, rows)) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(tile + sw128_offset(row, col + 8, rows)) = make_uint4(w[4], w[5], w[6], w[7]);
}

__device__ __forceinline__ void zero16_bf16(unsigned char* tile, int rows, int row, int col) {
  *reinterpret_cast<uint4*>(tile + sw128_offset(row, col, rows)) = make_uint4(0, 0, 0, 0);
  *reinterpret_cast<uint4*>(tile + sw128_offset(row, col + 8, rows)) = make_uint4(0, 0, 0, 0);
}

// TMA tile store shared -> global (rows outside the tensor are not written; coordinates
// must not be negative), its bulk-group commit, and the wait for the group's completion.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until the committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Same, but leaves the most recently committed group pending.
__device__ __forceinline__ void bulk_wait_read_prev() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// CTA barriers.  bar.sync counts whole warps, so a warp that reaches it with some lanes
// still inside a single-lane role (the TMA producer, the MMA issuer) would let the
// barrier complete early; every warp reconverges first.
__device__ __forceinline__ void cta_sync() {
  __syncwarp();
  __syncthreads();
}

// Named barrier over `n` threads (whole warps) of the CTA.
__device__ __forceinline__ void named_sync(int id, int n) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barrier over n threads that also returns whether v was true in any of them.
__device__ __forceinline__ bool named_sync_or(int id, int n, bool v) {
  __syncwarp();
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

}  // namespace tc
}  // namespace lz
