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
// Kernel: persistent, one CTA per SM walking 128 x 256 output tiles (128 rows
// of W, 256 tokens).  A TMA producer thread streams 64-wide K slices of W
// (K-major) and X (token-major rows, the "MN-major" operand, four 64-token
// boxes) into a 4-stage shared-memory ring of 48 KB stages with 128-byte
// swizzle; one thread issues tcgen05.mma (bf16 x bf16 -> fp32, M 128, N 256,
// K 16 per instruction) into one of two 256-column TMEM accumulators and
// releases each stage with tcgen05.commit; eight epilogue warps drain the other
// accumulator (warp w owns TMEM lanes 32 (w % 4) .. + 31, i.e. output rows,
// and 64 tokens of each half of the tile) into a swizzled bf16 staging tile of
// half the tile that a store warp writes out with bulk tensor stores, twice per
// tile, while the next tile accumulates.  The loads are latency bound (about
// 1.4 us per stage round trip out of L2): a 256-token tile reads W once for
// twice the outputs of a 128-token one, a quarter less traffic per output.  (A
// thread with bulk stores in flight stalls in its next proxy fence, so the
// fencing epilogue threads issue none.)  Every wait
// on an mbarrier is bounded: on expiry the kernel records SSM_ERR_TIMEOUT in
// the device status word (ssm_device_status), drains its outstanding copies
// with bounded waits, frees its TMEM and returns.
#include <cuda.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace ssm {

constexpr int kPM = 128;                       // output rows per tile (MMA M)
constexpr int kPN = 256;                       // tokens per tile (MMA N)
constexpr int kPK = 64;                        // K per stage: one 128-byte swizzle row of bf16
constexpr int kPStages = 4;
constexpr int kPEpiWarps = 8;                  // warps 0-7: epilogue (warp w: TMEM lane quadrant w % 4, column half w / 4)
constexpr int kPThreads = 32 * (kPEpiWarps + 3);   // + warp 8: TMA producer, warp 9: MMA issuer, warp 10: stores
constexpr int kPTileA = kPM * kPK * 2;         // 16 KB
constexpr int kPBox = kPK * 64 * 2;           // 8 KB: one 64-token box of X (64 K rows of 128 bytes)
constexpr int kPTileB = kPK * kPN * 2;         // 32 KB: four 64-token boxes
constexpr int kPStage = kPTileA + kPTileB;
constexpr int kPTileOut = kPM * (kPN / 2) * 2; // 32 KB: half the bf16 output tile, two 64-token boxes
constexpr int kPSmem = 1024 + kPStages * kPStage + kPTileOut + 256;   // slack, ring, staging, barriers
constexpr uint32_t kPTmemCols = 2 * kPN;       // two fp32 accumulators (one column per token)
constexpr uint32_t kProjIdesc = tc::idesc_bf16(kPM, kPN, false, true);   // A (W) K-major, B (X) MN-major

// device-side status of the asynchronous kernels (0 = fine, else an ssm_status)
__device__ int g_device_status = 0;

using namespace tc;

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
// The producer and the MMA issuer run ahead through a 4-stage shared-memory ring; two
// TMEM accumulators let the epilogue warps drain tile i while tile i + 1 accumulates.
__global__ void __launch_bounds__(kPThreads, 1)
proj_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 const __grid_constant__ CUtensorMap tmO, const ProjArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* stage_out = base + kPStages * kPStage;                 // kPTileOut
    uint64_t* full = reinterpret_cast<uint64_t*>(stage_out + kPTileOut);
    uint64_t* empty = full + kPStages;
    uint64_t* tfull = empty + kPStages;      // accumulator a ready for the epilogue
    uint64_t* tempty = tfull + 2;            // accumulator a drained by the epilogue
    uint64_t* ostaged = tempty + 2;          // the staging tile written (one buffer, [0] only; twice per tile)
    uint64_t* ofree = ostaged + 2;           // ... and read out by its bulk stores
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ofree + 2);
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
            mbar_init(&ostaged[q], kPEpiWarps);
            mbar_init(&ofree[q], 1);
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
            // producer: K slices of W (rows m0..m0+127) and of X[b] (tokens n0..n0+255)
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
#pragma unroll
                    for (int j = 0; j < kPN / 64; j++)
                        tma_load_3d(st + kPTileA + j * kPBox, &tmX, &full[s], n0 + 64 * j, kb * kPK, bz);
                }
            }
            // copies still in flight must land before the CTA may exit
            for (int u = (it > kPStages ? it - kPStages : 0); u < it; u++) mbar_wait(&full[u % kPStages], (u / kPStages) & 1);
        }
    } else if (warp == kPEpiWarps + 1) {
        if (lane == 0) {
            // MMA issuer; descriptors of stage 0 built once (stage s is s * kPStage bytes further)
            const uint64_t dA0 = sw128_desc(smem_addr(base), 16, 1024);
            const uint64_t dB0 = sw128_desc(smem_addr(base + kPTileA), kPBox, 1024);
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
#pragma unroll
                    for (int k = 0; k < kPK / 16; k++) {
                        // A: K-major rows of 128 bytes, 8-row groups 1024 bytes apart; the
                        // K step of 16 elements is 32 bytes along the swizzled row.
                        // B: token-major rows of 128 bytes (64 tokens), 8-row groups of K
                        // 1024 bytes apart, each next 64 tokens 8 KB further; the K step
                        // of 16 rows is 2 KB.
                        const uint64_t so = (uint64_t)(s * (kPStage >> 4));
                        umma_bf16(dcol, dA0 + so + kmajor_step(k, 0), dB0 + so + mnmajor_step(k), kProjIdesc,
                                  (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(&empty[s]);   // the stage is free once these MMAs have read it
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
            }
        }
    } else if (warp == kPEpiWarps + 2) {
        if (lane == 0) {
            // stores: each staged half tile leaves by two bulk tensor stores; this thread issues
            // no proxy fences, so no fence elsewhere waits for the stores in flight
            int use = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < a.tiles && ok; tile += gridDim.x) {
                int m0, n0, bz;
                tile_coords(a, tile, m0, n0, bz);
                for (int hs = 0; hs < 2; hs++, use++) {
                    if (!mbar_wait(&ostaged[0], use & 1)) {
                        record_timeout(abort_flag);
                        ok = false;
                        break;
                    }
                    tma_store_3d(&tmO, stage_out, n0 + 128 * hs, m0, bz);
                    tma_store_3d(&tmO, stage_out + kPTileOut / 2, n0 + 128 * hs + 64, m0, bz);
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                    mbar_arrive(&ofree[0]);
                }
            }
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        }
    } else {
        // epilogue: warp w reads TMEM lanes (output rows) 32 (w % 4) .. + 31 and, of each
        // 128-token half of the tile, tokens 64 (w / 4) .. + 63
        const int quad = warp & 3, half = warp >> 2;
        int use = 0;   // staging-tile uses so far (two per tile)
        int local = 0;
        for (int tile = blockIdx.x; tile < a.tiles; tile += gridDim.x, local++) {
            const int acc = local & 1;
            // one decision for all epilogue warps (tcgen05.ld needs whole warps, and
            // the named barriers below need all of them)
            const bool waited = mbar_wait(&tfull[acc], (local >> 1) & 1);
            if (!waited) record_timeout(abort_flag);
            if (!epi_all(waited && *(volatile int*)abort_flag == 0)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            int m0, n0, bz;
            tile_coords(a, tile, m0, n0, bz);
            const int row = m0 + quad * 32 + lane;
            const float bias = (a.bias != nullptr && row < a.m) ? __ldg(a.bias + row) : 0.f;
            // w[2 hs + c]: half tile hs, 32-token chunk c of this warp's 64
            uint32_t w[4][16];
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t r[32];
                const int col = 128 * (c >> 1) + 64 * half + 32 * (c & 1);
                tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * kPN + col), r);
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    float v0 = __uint_as_float(r[2 * i]) + bias, v1 = __uint_as_float(r[2 * i + 1]) + bias;
                    if (a.epilogue == 1) {
                        // SFU softplus: error near 1e-6 relative, far below the bf16 rounding that follows
                        v0 = softplus_fast(v0);
                        v1 = softplus_fast(v1);
                    }
                    w[c][i] = pack_bf16x2(v0, v1);
                }
            }
            // the accumulator is in registers: hand it back to the MMA warp
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&tempty[acc])) : "memory");
            // stage each half of the tile (128-byte swizzled rows, two 64-token boxes) for the
            // store warp; the staging tile must have been read out by its previous store
            const int rt = quad * 32 + lane;   // row within the tile
            bool live = true;
#pragma unroll
            for (int hs = 0; hs < 2; hs++, use++) {
                const bool freed = use < 1 || mbar_wait(&ofree[0], (use - 1) & 1);
                if (!freed) record_timeout(abort_flag);
                if (!epi_all(freed && *(volatile int*)abort_flag == 0)) {
                    live = false;
                    break;
                }
#pragma unroll
                for (int c = 0; c < 2; c++) {
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const int ch = 4 * c + q;   // 16-byte chunk of this warp's 64-token box
                        *reinterpret_cast<uint4*>(stage_out + half * (kPTileOut / 2) + rt * 128 + ((ch ^ (rt & 7)) << 4)) =
                            make_uint4(w[2 * hs + c][4 * q], w[2 * hs + c][4 * q + 1], w[2 * hs + c][4 * q + 2],
                                       w[2 * hs + c][4 * q + 3]);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&ostaged[0]);
            }
            if (!live) break;
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == kPEpiWarps + 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps, then one launch.

cudaError_t launch_proj(const ssm_proj_params* p, cudaStream_t st) {
    alignas(64) CUtensorMap tmW, tmX, tmO;
    cudaError_t e;
    {
        const uint64_t dims[2] = {(uint64_t)p->k, (uint64_t)p->m};
        const uint64_t strides[1] = {(uint64_t)p->ldw * 2};
        const uint32_t box[2] = {(uint32_t)kPK, (uint32_t)kPM};
        if ((e = encode_bf16_map(&tmW, p->W, 2, dims, strides, box, true, true)) != cudaSuccess) return e;
    }
    // with one batch row the batch stride is never used: give the maps a valid one
    const int64_t xbs = p->batch > 1 ? p->x_batch_stride : p->ldx * p->k;
    const int64_t obs = p->batch > 1 ? p->out_batch_stride : p->ldo * p->m;
    {
        const uint64_t dims[3] = {(uint64_t)p->n, (uint64_t)p->m, (uint64_t)p->batch};
        const uint64_t strides[2] = {(uint64_t)p->ldo * 2, (uint64_t)obs * 2};
        const uint32_t box[3] = {64, (uint32_t)kPM, 1};
        if ((e = encode_bf16_map(&tmO, p->out, 3, dims, strides, box, true, false)) != cudaSuccess) return e;
    }
    {
        const uint64_t dims[3] = {(uint64_t)p->n, (uint64_t)p->k, (uint64_t)p->batch};
        const uint64_t strides[2] = {(uint64_t)p->ldx * 2, (uint64_t)xbs * 2};
        const uint32_t box[3] = {64, (uint32_t)kPK, 1};
        if ((e = encode_bf16_map(&tmX, p->X, 3, dims, strides, box, true, true)) != cudaSuccess) return e;
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

namespace tc {
cudaError_t device_status_word(int** ptr) {
    void* a = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&a, g_device_status);
    *ptr = static_cast<int*>(a);
    return e;
}
}  // namespace tc

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
