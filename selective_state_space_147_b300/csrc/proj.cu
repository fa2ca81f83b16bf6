// proj.cu -- the dense projections beside the selective scan on the tensor
// cores: x_proj (conv output -> [dt_raw, B, C]) and dt_proj (dt_raw -> delta),
// sm_103a.
//
// "Mamba 模型" (gaos6e.github.io), block flowchart: the conv output Xc_t feeds
// the x_proj node, which produces dt_raw_t, B_t and C_t, and dt_raw_t feeds the
// dt_proj + softplus node, which produces delta_t.  Both are matrix products
// with weights shared by every token:  out[b] (M x T) = W (M x K) X[b] (K x T),
// where X[b] is channel-major with the tokens contiguous -- the layout the scan
// reads -- so the outputs land directly in the scan's layouts: x_proj's rows
// [R, R+N) and [R+N, R+2N) are B and C as (batch, N, L) views, its first R
// rows are dt_proj's input, and dt_proj writes delta as (batch, D, L).
//
// Kernel: persistent, one CTA per SM walking 128 x 128 output tiles.  A TMA
// producer thread streams 64-wide K slices of W (K-major) and X (token-major
// rows, the "MN-major" operand) into a 6-stage shared-memory ring with 128-byte
// swizzle; one thread issues tcgen05.mma (bf16 x bf16 -> fp32, M 128, N 128,
// K 16 per instruction) into one of two TMEM accumulators and releases each
// stage with tcgen05.commit; four epilogue warps drain the other accumulator
// (warp w owns TMEM lanes 32w..32w+31, i.e. output rows) into a swizzled
// bf16 tile in shared memory that one thread writes out with bulk tensor
// stores, while the next tile accumulates.  Every wait
// on an mbarrier is bounded: on expiry the kernel records SSM_ERR_TIMEOUT in
// the device status word (ssm_device_status), drains its outstanding copies
// with bounded waits, frees its TMEM and returns.
#include <cuda.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace ssm {

constexpr int kPM = 128;                       // output rows per tile (MMA M)
constexpr int kPN = 128;                       // tokens per tile (MMA N)
constexpr int kPK = 64;                        // K per stage: one 128-byte swizzle row of bf16
constexpr int kPStages = 4;
constexpr int kPEpiWarps = 4;                  // warps 0-3: epilogue (TMEM lane quadrants 0-3)
constexpr int kPThreads = 32 * (kPEpiWarps + 2);   // + warp 4: TMA producer, warp 5: MMA issuer
constexpr int kPTileA = kPM * kPK * 2;         // 16 KB
constexpr int kPTileB = kPK * kPN * 2;         // 16 KB: two 64-token boxes of 8 KB
constexpr int kPStage = kPTileA + kPTileB;
constexpr int kPTileOut = kPM * kPN * 2;       // 32 KB: the bf16 output tile, two 64-token boxes
constexpr int kPSmem = 1024 + kPStages * kPStage + 2 * kPTileOut + 256;   // slack, ring, staging, barriers
constexpr uint32_t kPTmemCols = 2 * kPN;       // two fp32 accumulators (one column per token)
constexpr long long kWaitLimit = 4000000000LL; // cycles (about 2 s) before a wait gives up

// device-side status of the asynchronous kernels (0 = fine, else an ssm_status)
__device__ int g_device_status = 0;

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
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

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(smem_addr(dst)), "l"(map), "r"(smem_addr(bar)), "r"(x), "r"(y)
        : "memory");
}
// bulk tensor store of a staged shared-memory box (completion tracked by bulk groups)
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(map),
                 "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
        "[%2];" ::"r"(smem_addr(dst)),
        "l"(map), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// Shared-memory matrix descriptor of a 128-byte-swizzled operand tile:
// start address, leading and stride byte offsets (all >> 4), the descriptor
// version of this architecture and the swizzle mode.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version
    d |= (uint64_t)2 << 61;   // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B MN-major (token-contiguous rows), N >> 3 and M >> 4.
constexpr uint32_t kProjIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                                ((uint32_t)(kPN >> 3) << 17) | ((uint32_t)(kPM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(kProjIdesc), "r"(accumulate)
        : "memory");
}
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

struct ProjArgs {
    int64_t m, n, k;
    __nv_bfloat16* out;
    int64_t ldo, out_bs;
    const float* bias;
    int epilogue;   // 0: acc (+ bias); 1: softplus(acc + bias)
    int mt, nt, tiles;   // tile counts: rows, tokens, all (rows fastest, then tokens, then batch)
};

__device__ __forceinline__ void tile_coords(const ProjArgs& a, int tile, int& m0, int& n0, int& bz) {
    const int mi = tile % a.mt;
    const int rest = tile / a.mt;
    m0 = mi * kPM;
    n0 = (rest % a.nt) * kPN;
    bz = rest / a.nt;
}

// AND of v over the 128 epilogue threads (named barrier 1); every epilogue thread must call it
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(r)
                 : "r"((uint32_t)v), "n"(32 * kPEpiWarps)
                 : "memory");
    return r != 0;
}

__device__ __forceinline__ void record_timeout(int* abort_flag) {
    atomicExch(&g_device_status, (int)SSM_ERR_TIMEOUT);
    *(volatile int*)abort_flag = 1;
}

// Persistent: every CTA (one per SM) walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// The producer and the MMA issuer run ahead through a 6-stage shared-memory ring; two
// TMEM accumulators let the epilogue warps drain tile i while tile i + 1 accumulates.
__global__ void __launch_bounds__(kPThreads, 1)
proj_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 const __grid_constant__ CUtensorMap tmO, const ProjArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* stage_out = base + kPStages * kPStage;                 // 2 x kPTileOut
    uint64_t* full = reinterpret_cast<uint64_t*>(stage_out + 2 * kPTileOut);
    uint64_t* empty = full + kPStages;
    uint64_t* tfull = empty + kPStages;      // accumulator a ready for the epilogue
    uint64_t* tempty = tfull + 2;            // accumulator a drained by the epilogue
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nk = (int)((a.k + kPK - 1) / kPK);

    if (tid == 0) {
        for (int s = 0; s < kPStages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int q = 0; q < 2; q++) {
            mbar_init(&tfull[q], 1);
            mbar_init(&tempty[q], kPEpiWarps);   // one arrival per epilogue warp
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kPEpiWarps + 1) {   // the MMA warp allocates (and later frees) the accumulators
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kPTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == kPEpiWarps) {
        if (lane == 0) {
            // producer: K slices of W (rows m0..m0+127) and of X[b] (tokens n0..n0+127)
            int it = 0;   // stage uses so far
            for (int tile = blockIdx.x; tile < a.tiles && !*(volatile int*)abort_flag; tile += gridDim.x) {
                int m0, n0, bz;
                tile_coords(a, tile, m0, n0, bz);
                for (int kb = 0; kb < nk; kb++, it++) {
                    const int s = it % kPStages;
                    if (it >= kPStages && !mbar_wait(&empty[s], ((it / kPStages) - 1) & 1)) {
                        record_timeout(abort_flag);
                        break;
                    }
                    unsigned char* st = base + s * kPStage;
                    mbar_expect_tx(&full[s], kPStage);
                    tma_load_2d(st, &tmW, &full[s], kb * kPK, m0);
                    tma_load_3d(st + kPTileA, &tmX, &full[s], n0, kb * kPK, bz);
                    tma_load_3d(st + kPTileA + kPTileB / 2, &tmX, &full[s], n0 + 64, kb * kPK, bz);
                }
            }
            // copies still in flight must land before the CTA may exit
            for (int u = (it > kPStages ? it - kPStages : 0); u < it; u++) mbar_wait(&full[u % kPStages], (u / kPStages) & 1);
        }
    } else if (warp == kPEpiWarps + 1) {
        if (lane == 0) {
            // MMA issuer
            int it = 0, local = 0;
            for (int tile = blockIdx.x; tile < a.tiles; tile += gridDim.x, local++) {
                if (*(volatile int*)abort_flag) break;
                const int acc = local & 1;
                if (local >= 2 && !mbar_wait(&tempty[acc], ((local >> 1) - 1) & 1)) {
                    record_timeout(abort_flag);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t dcol = tmem + (uint32_t)(acc * kPN);
                bool ok = true;
                for (int kb = 0; kb < nk; kb++, it++) {
                    const int s = it % kPStages;
                    if (!mbar_wait(&full[s], (it / kPStages) & 1)) {
                        record_timeout(abort_flag);
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t sa = smem_addr(base + s * kPStage);
                    const uint32_t sb = sa + kPTileA;
#pragma unroll
                    for (int k = 0; k < kPK / 16; k++) {
                        // A: K-major rows of 128 bytes, 8-row groups 1024 bytes apart; the
                        // K step of 16 elements is 32 bytes along the swizzled row.
                        // B: token-major rows of 128 bytes (64 tokens), 8-row groups of K
                        // 1024 bytes apart, the second 64 tokens 8 KB further; the K step
                        // of 16 rows is 2 KB.
                        umma_bf16(dcol, sw128_desc(sa + 32 * k, 16, 1024), sw128_desc(sb + 2048 * k, kPTileB / 2, 1024),
                                  (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(&empty[s]);   // the stage is free once these MMAs have read it
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
            }
        }
    } else {
        // epilogue: warp w reads TMEM lanes (output rows) 32w .. 32w + 31
        int local = 0;
        for (int tile = blockIdx.x; tile < a.tiles; tile += gridDim.x, local++) {
            const int acc = local & 1;
            // one decision for all four epilogue warps (tcgen05.ld needs whole warps,
            // and the named barriers below need all four)
            const bool waited = mbar_wait(&tfull[acc], (local >> 1) & 1);
            if (!waited) record_timeout(abort_flag);
            if (!epi_all(waited && *(volatile int*)abort_flag == 0)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            int m0, n0, bz;
            tile_coords(a, tile, m0, n0, bz);
            const int row = m0 + warp * 32 + lane;
            const float bias = (a.bias != nullptr && row < a.m) ? __ldg(a.bias + row) : 0.f;
            uint32_t w[4][16];
#pragma unroll
            for (int c = 0; c < kPN / 32; c++) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(acc * kPN + c * 32), r);
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    float v0 = __uint_as_float(r[2 * i]) + bias, v1 = __uint_as_float(r[2 * i + 1]) + bias;
                    if (a.epilogue == 1) {
                        v0 = v0 > 20.f ? v0 : log1pf(expf(v0));
                        v1 = v1 > 20.f ? v1 : log1pf(expf(v1));
                    }
                    w[c][i] = pack_bf16x2(v0, v1);
                }
            }
            // the accumulator is in registers: hand it back to the MMA warp
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&tempty[acc])) : "memory");
            // stage the tile (128-byte swizzled rows, two 64-token boxes) for one bulk store;
            // the staging buffer used two tiles ago must have been read out first
            unsigned char* so = stage_out + (local & 1) * kPTileOut;
            if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kPEpiWarps) : "memory");
            const int rt = warp * 32 + lane;   // row within the tile
#pragma unroll
            for (int c = 0; c < kPN / 32; c++) {
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const int col = 32 * c + 8 * q;            // first token of this 16-byte chunk
                    const int box = col >> 6, ch = (col & 63) >> 3;
                    *reinterpret_cast<uint4*>(so + box * (kPTileOut / 2) + rt * 128 + ((ch ^ (rt & 7)) << 4)) =
                        make_uint4(w[c][4 * q], w[c][4 * q + 1], w[c][4 * q + 2], w[c][4 * q + 3]);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kPEpiWarps) : "memory");
            if (tid == 0) {
                tma_store_3d(&tmO, so, n0, m0, bz);
                tma_store_3d(&tmO, so + kPTileOut / 2, n0 + 64, m0, bz);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
        }
        if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == kPEpiWarps + 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps through the driver's entry point (the library does not
// link the driver library), then one launch.

typedef CUresult (*PfnEncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static cudaError_t encode_fn(PfnEncodeTiled* out) {
    static PfnEncodeTiled fn = nullptr;
    if (fn == nullptr) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || f == nullptr) return cudaErrorSymbolNotFound;
        fn = reinterpret_cast<PfnEncodeTiled>(f);
    }
    *out = fn;
    return cudaSuccess;
}

cudaError_t launch_proj(const ssm_proj_params* p, cudaStream_t st) {
    PfnEncodeTiled enc = nullptr;
    cudaError_t e = encode_fn(&enc);
    if (e != cudaSuccess) return e;
    alignas(64) CUtensorMap tmW, tmX;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p->k, (cuuint64_t)p->m};
        const cuuint64_t strides[1] = {(cuuint64_t)p->ldw * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kPK, (cuuint32_t)kPM};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p->W), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // with one batch row the batch stride is never used: give the maps a valid one
    const int64_t xbs = p->batch > 1 ? p->x_batch_stride : p->ldx * p->k;
    const int64_t obs = p->batch > 1 ? p->out_batch_stride : p->ldo * p->m;
    alignas(64) CUtensorMap tmO;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)p->n, (cuuint64_t)p->m, (cuuint64_t)p->batch};
        const cuuint64_t strides[2] = {(cuuint64_t)p->ldo * 2, (cuuint64_t)obs * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)kPM, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tmO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p->out, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)p->n, (cuuint64_t)p->k, (cuuint64_t)p->batch};
        const cuuint64_t strides[2] = {(cuuint64_t)p->ldx * 2, (cuuint64_t)xbs * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)kPK, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p->X), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    ProjArgs a;
    a.m = p->m; a.n = p->n; a.k = p->k;
    a.out = static_cast<__nv_bfloat16*>(p->out);
    a.ldo = p->ldo; a.out_bs = p->out_batch_stride;
    a.bias = p->bias;
    a.epilogue = p->epilogue;
    a.mt = (int)ceil_div(p->m, (int64_t)kPM);
    a.nt = (int)ceil_div(p->n, (int64_t)kPN);
    const int64_t tiles = (int64_t)a.mt * a.nt * p->batch;
    if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
    a.tiles = (int)tiles;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = prepare_kernel<proj_gemm_kernel>(kPSmem);
    if (e != cudaSuccess) return e;
    const int grid = (int)(tiles < sms ? tiles : sms);
    proj_gemm_kernel<<<grid, kPThreads, kPSmem, st>>>(tmW, tmX, tmO, a);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t read_device_status(int* status, int clear) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
    if (e != cudaSuccess) return e;
    *status = v;
    if (clear && v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
    }
    return e;
}

}  // namespace ssm
