// tc.cuh -- the Blackwell tensor-core plumbing shared by the kernels that use
// it (projections, SSD chunks): mbarriers with bounded waits, TMA tile copies
// (cp.async.bulk.tensor), shared-memory matrix descriptors for 128-byte
// swizzled tiles, tcgen05.mma issue / commit and TMEM loads, plus the host
// helper that encodes a bf16 tensor map through the driver's entry point.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ssm.h"

namespace ssm {
namespace tc {

constexpr long long kWaitLimit = 4000000000LL;   // cycles (about 2 s) before a wait gives up

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Wait until the phase of parity `parity` has completed; false after kWaitLimit cycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_addr(bar);
    const long long t0 = clock64();
    while (true) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > kWaitLimit) return false;
    }
}

// true if the phase of parity `parity` has completed (does not wait)
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(smem_addr(dst)), "l"(map), "r"(smem_addr(bar)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
        "[%2];" ::"r"(smem_addr(dst)),
        "l"(map), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, "
        "%6}], [%2];" ::"r"(smem_addr(dst)),
        "l"(map), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}
// bulk tensor store of a staged shared-memory box (completion tracked by bulk groups)
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(map),
                 "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Shared-memory matrix descriptor of a 128-byte-swizzled operand tile:
// start address, leading and stride byte offsets (all >> 4), the descriptor
// version of this architecture and the swizzle mode.  K-major operands: rows
// of 128 bytes (64 bf16 along K), 8-row groups `sbo` apart, the K step of 16
// elements advances the start by 32 bytes.  MN-major operands: rows of 64
// consecutive M (or N) elements, one row per K index, 8-row groups `sbo`
// apart, the next 64 M (or N) elements `lbo` further; the K step of 16 rows
// advances the start by 2 KB.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version
    d |= (uint64_t)2 << 61;   // 128-byte swizzle
    return d;
}

// Start-address offsets (16-byte units, added to a descriptor) of the K step k
// of 16 elements: K-major tiles of 64-wide atoms `atom_bytes` apart, and
// MN-major tiles (16 rows of 128 bytes per step).  The issuing thread adds
// these to descriptors built once, so a tcgen05.mma costs it a few
// instructions: built per instruction, descriptors made the issue rate, not
// the tensor core, the bound.
__host__ __device__ constexpr uint64_t kmajor_step(int k, int atom_bytes) {
    return (uint64_t)(((k >> 2) * atom_bytes + (k & 3) * 32) >> 4);
}
__host__ __device__ constexpr uint64_t mnmajor_step(int k) { return (uint64_t)(k * 128); }

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, the
// major-ness of each operand (true = MN-major), N >> 3 and M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D (TMEM) (+)= A (smem) B (smem), issued by one thread.  Each descriptor is
// passed as its two 32-bit halves and assembled into a 64-bit register inside
// the instruction's own asm block: the high half is a per-operand constant
// (stride offsets, version, swizzle), the low half the start address (plus
// the leading offset), so a K step is one 32-bit add.  (With both 64-bit
// descriptors held in registers across the issuing loop, products that shared
// an A descriptor with an earlier one read the wrong B operand.)
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n .reg .b64 ad, bd;\n mov.b64 ad, {%1, %2};\n mov.b64 bd, {%3, %4};\n"
        " setp.ne.b32 p, %6, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p;\n}\n"
        ::"r"(tmem_d), "r"((uint32_t)adesc), "r"((uint32_t)(adesc >> 32)), "r"((uint32_t)bdesc),
        "r"((uint32_t)(bdesc >> 32)), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D (TMEM) (+)= A (TMEM) B (smem): A in tensor memory as K-major rows, one row per TMEM
// lane, two bf16 K elements per 32-bit column (the lower element in the low half); the
// K step of 16 elements is 8 columns.
__device__ __forceinline__ void umma_bf16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n .reg .b64 bd;\n mov.b64 bd, {%2, %3};\n setp.ne.b32 p, %5, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n}\n"
        ::"r"(tmem_d), "r"(tmem_a), "r"((uint32_t)bdesc), "r"((uint32_t)(bdesc >> 32)), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on `bar` once every tcgen05.mma issued so far by this thread has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane; tmem_st_wait() before they are read
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes become visible to the tensor core / TMA
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// host: a tiled tensor map (rank <= 5) of bf16 (or fp32 with `fp32`); strides
// in bytes for dimensions 1..rank-1
cudaError_t encode_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128, bool l2_promote,
                       bool fp32);
inline cudaError_t encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                                   const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128,
                                   bool l2_promote) {
    return encode_map(map, base, rank, dims, strides_bytes, box, swizzle128, l2_promote, false);
}

// host: the address of the device status word the asynchronous kernels record
// SSM_ERR_TIMEOUT in (0 = fine)
cudaError_t device_status_word(int** ptr);

}  // namespace tc
}  // namespace ssm
