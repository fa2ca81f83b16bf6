// ssd.cu -- Mamba-2 state-space-duality (SSD) layer, forward, sm_103a.
//
// Method ("Mamba 与状态空间模型", section 09 "Mamba-2：两种算法"; pnsm.cn overview,
// section "Mamba-2：状态空间对偶性", chunked algorithm): A is one number per head
// times the identity, so the layer is a product with a lower-triangular matrix
// whose (i, j) entry is C_i . B_j times the decay between steps j and i.  The
// sequence is cut into chunks: inside a chunk that product is evaluated with
// matrix multiplications on the tensor cores, between chunks only the state
// (N x P per head) is passed on.  Per (batch b, head h), chunk of Q = 128
// steps starting at t0, with Delta_t = softplus(dt + dt_bias), s_i =
// sum_{r<=i} Delta_r A (inclusive, inside the chunk) and H the state entering
// the chunk:
//
//   y_i = exp(s_i) C_i^T H                                    (inter-chunk)
//       + sum_{j<=i} (C_i . B_j) exp(s_i - s_j) Delta_j x_j   (intra-chunk)
//       + D x_i
//   H'  = exp(s_last) H + sum_j exp(s_last - s_j) Delta_j B_j x_j^T
//
// Design for B300: one CTA per (b, h) walks the chunks in order; every
// contraction is a tcgen05.mma (bf16 x bf16 -> fp32 in TMEM, M = 128 rows):
//   G  = C B^T           (128 x 128, K = N)           A = C tile, B = B tile (both K-major)
//   Yd = M X             (128 x 64,  K = 128 steps)   M = G o decay o Delta (lower triangle),
//                                                     written to TMEM and read from there
//   S  = B^T (w o X)     (N x 64,    K = 128 steps)   A = the B tile read state-major
//   Yo = C H             (128 x 64,  K = N)           H = the entering state in bf16
// y = Yd + exp(s_i) Yo + D x, and the fp32 state H' = exp(s_last) H + S stays in
// the epilogue threads' registers across chunks (its bf16 copy is the next
// chunk's operand).  Warp 8 streams the C, B and x tiles of a chunk with TMA
// (128-byte swizzle; rows past the sequence end and states past N read as
// zero) into a 2-stage ring and computes each chunk's Delta and in-chunk prefix
// sums s ahead of time; warp 9 issues the MMAs -- C H while the epilogue warps
// build w o X, B^T (w o X) while they turn G into M, the next chunk's G after
// M X -- and eight epilogue warps (warp w: TMEM lanes 32 (w % 4) .. + 31 = chunk
// rows, half w / 4 of the columns) compute w o X into shared memory and M into
// tensor memory (exp per element only in the diagonal 32 x 32 blocks; below them the decay
// factors into exp(s_i - s_e) exp(s_e - s_j), both exponents <= 0), then the
// state update and y, which leaves through a swizzled staging tile and bulk
// tensor stores that warp 10 issues (a thread with bulk stores in flight would
// stall in its next proxy fence, so the fencing epilogue threads issue none).  Every mbarrier wait is bounded: on
// expiry the kernel records SSM_ERR_TIMEOUT in the device status word and the
// CTA leaves after its own copies and MMAs have landed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace ssm {

namespace {

using namespace tc;

constexpr int kQ = 128;                   // chunk length: the MMA's M (rows = steps)
constexpr int kP = 64;                    // head dimension
constexpr int kAtom = 128 * 128;          // 16 KB: 128 rows of 128 bytes (64 bf16)
constexpr int kTileBC = 2 * kAtom;        // a C or B tile: 128 steps x 128 states (two 64-state atoms)
constexpr int kTileX = kAtom;             // an x tile: 128 steps x 64 head-dimension columns
constexpr int kStage = 2 * kTileBC + kTileX;
constexpr int kStages = 2;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (kEpiWarps + 3);   // + warp 8: TMA producer, warp 9: MMA issuer, warp 10: output stores
constexpr int kOffM = kStages * kStage;           // the output staging tile (y of a chunk)
constexpr int kOffWX = kOffM + 2 * kAtom;         // w o x: MN-major B operand
constexpr int kOffH = kOffWX + kTileX;            // the entering state in bf16: MN-major B operand
constexpr int kOffAux = kOffH + kTileX;
// aux: Delta[2][128], s[2][128] (fp32, double-buffered by chunk parity), the column factors of
// the blocks below M's diagonal [128], barriers
constexpr int kAuxFloats = 2 * kQ * 2 + kQ;
// full, empty (C and B), fullx, emptyx (x), dready, gfull, wready, mready, yfull, yempty, done, ystaged, yfree
constexpr int kNumBars = 2 + 2 + 2 + 2 + 2 + 2 + 1 + 1 + 1 + 1 + 1 + 1 + 1 + 1;
constexpr int kSmem = kOffAux + kAuxFloats * 4 + kNumBars * 8 + 16;
// TMEM columns: G (two buffers), Yd, Yo, S, and M (bf16, two per column: Yd's A operand)
constexpr uint32_t kColG = 0, kColYd = 256, kColYo = 320, kColS = 384, kColM = 448, kTmemCols = 512;

struct SsdArgs {
    int L, H, heads_per_group, nstate, nbox, nchunks;
    uint32_t cb_bytes;   // C and B bytes of one stage (64 or 128 states per tile row)
    const __nv_bfloat16* dt;     // (batch, L, H)
    const float* A;              // (H)
    const float* D;              // (H) or NULL
    const float* dt_bias;        // (H) or NULL
    const float* h0;             // (batch, H, N, P) or NULL
    float* final_state;          // (batch, H, N, P) or NULL
    void* out;                   // (batch, L, H, P)
    int softplus;
    int* status;                 // device status word
};

__device__ __forceinline__ void record_timeout(int* status, int* abort_flag) {
    atomicExch(status, (int)SSM_ERR_TIMEOUT);
    *(volatile int*)abort_flag = 1;
}

// AND of v over the 256 epilogue threads (named barrier 1); every epilogue thread must call it
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(r)
                 : "r"((uint32_t)v), "n"(32 * kEpiWarps)
                 : "memory");
    return r != 0;
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}

// the 16-byte chunk `ch` of row `r` of a 128-byte-swizzled tile
__device__ __forceinline__ unsigned char* swz(unsigned char* tile, int r, int ch) {
    return tile + r * 128 + ((ch ^ (r & 7)) << 4);
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
ssd_chunk_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY, const SsdArgs a) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the swizzled tiles need a 1024-byte aligned base: refuse (uniformly) otherwise
    if (smem_addr(smem) & 1023) {
        if (tid == 0) atomicExch(a.status, (int)SSM_ERR_MISALIGNED);
        return;
    }
    float* dl = reinterpret_cast<float*>(smem + kOffAux);   // Delta [2][128]
    float* s2 = dl + 2 * kQ;                                  // s log2(e) [2][128]
    float* cf = s2 + 2 * kQ;                                  // [128]
    uint64_t* full = reinterpret_cast<uint64_t*>(cf + kQ);   // C and B tiles of stage s landed
    uint64_t* empty = full + 2;                               // ... and read by the chunk's C H and B^T (w o x)
    uint64_t* fullx = empty + 2;                              // the x tile of stage s landed
    uint64_t* emptyx = fullx + 2;                             // ... and read by the chunk's M x
    uint64_t* dready = emptyx + 2;  // Delta and s of chunk c in buffer c & 1
    uint64_t* gfull = dready + 2;
    uint64_t* wready = gfull + 2;
    uint64_t* mready = wready + 1;
    uint64_t* yfull = mready + 1;
    uint64_t* yempty = yfull + 1;
    uint64_t* done = yempty + 1;
    uint64_t* ystaged = done + 1;   // the output tile of a chunk is in its staging buffer
    uint64_t* yfree = ystaged + 1;  // ... and has been read out by its bulk store
    uint64_t* sfull = yfree + 1;    // S of the chunk (and its C H before it) complete
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sfull + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int unit = blockIdx.x;
    const int b = unit / a.H, h = unit % a.H, g = h / a.heads_per_group;
    const int nc = a.nchunks;

    if (tid == 0) {
        for (int s = 0; s < 2; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&fullx[s], 1);
            mbar_init(&emptyx[s], 1);
            mbar_init(&dready[s], 1);
            mbar_init(&gfull[s], 1);
        }
        mbar_init(wready, kEpiWarps);
        mbar_init(mready, kEpiWarps);
        mbar_init(yfull, 1);
        mbar_init(yempty, kEpiWarps);
        mbar_init(done, 1);
        mbar_init(ystaged, kEpiWarps);
        mbar_init(yfree, 1);
        mbar_init(sfull, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kEpiWarps + 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == kEpiWarps) {
        // producer warp: lane 0 streams each chunk's C, B (state boxes of 64) and x tiles into
        // stage c & 1; then the warp computes the chunk's Delta and in-chunk prefix sums of
        // Delta A (log2 units), four consecutive steps per lane, into buffer c & 1.
        const float Al2 = __ldg(a.A + h) * kLog2e;
        const float bias = a.dt_bias != nullptr ? __ldg(a.dt_bias + h) : 0.f;
        // the raw step sizes of a chunk are loaded one chunk ahead (their latency is long
        // next to the tile traffic, and nothing here waits on them early)
        auto load_dt = [&](int c, float (&r)[4]) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int t = c * kQ + 4 * lane + i;
                r[i] = t < a.L ? __bfloat162float(a.dt[((size_t)b * a.L + t) * a.H + h]) : 0.f;
            }
        };
        int issued = 0;
        // one chunk: its C and B tiles into stage c & 1 once chunk c - 2's C H and B^T (w o x)
        // have read them, its x tile once chunk c - 2's M x has, then its Delta and s into
        // buffer c & 1 from the raw step sizes `cur`, while the next chunk's load into `nxt`.
        // Buffer c & 1 was last read by chunk c - 2's decay matrix, finished before its M x.
        auto step = [&](int c, const float (&cur)[4], float (&nxt)[4]) -> bool {
            const int s = c & 1;
            int go = 1;
            if (lane == 0) {
                if (c >= 2 && !mbar_wait(&empty[s], ((c >> 1) - 1) & 1)) {
                    record_timeout(a.status, abort_flag);
                    go = 0;
                }
                if (go && *(volatile int*)abort_flag) go = 0;
                unsigned char* st = smem + s * kStage;
                if (go) {
                    mbar_expect_tx(&full[s], a.cb_bytes);
                    for (int bx = 0; bx < a.nbox; bx++) {
                        tma_load_4d(st + bx * kAtom, &tmC, &full[s], 64 * bx, g, c * kQ, b);
                        tma_load_4d(st + kTileBC + bx * kAtom, &tmB, &full[s], 64 * bx, g, c * kQ, b);
                    }
                    issued = c + 1;
                }
                if (go && c >= 2 && !mbar_wait(&emptyx[s], ((c >> 1) - 1) & 1)) {
                    record_timeout(a.status, abort_flag);
                    go = 0;
                }
                if (go) {
                    mbar_expect_tx(&fullx[s], kTileX);
                    tma_load_3d(st + 2 * kTileBC, &tmX, &fullx[s], h * kP, c * kQ, b);
                }
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) return false;
            if (c + 1 < nc) load_dt(c + 1, nxt);
            float dv[4], av[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int t = c * kQ + 4 * lane + i;
                dv[i] = 0.f;
                if (t < a.L) {
                    const float v = cur[i] + bias;
                    // SFU softplus (~1e-6 relative): far inside the bf16 roundings of the chunked
                    // algorithm, and cheaper than the library form on this warp's path
                    dv[i] = a.softplus ? softplus_fast(v) : v;
                }
                av[i] = dv[i] * Al2 + (i > 0 ? av[i - 1] : 0.f);
            }
            float tot = av[3];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, tot, o);
                if (lane >= o) tot += y;
            }
            const float off = tot - av[3];
            *reinterpret_cast<float4*>(dl + s * kQ + 4 * lane) = make_float4(dv[0], dv[1], dv[2], dv[3]);
            *reinterpret_cast<float4*>(s2 + s * kQ + 4 * lane) =
                make_float4(av[0] + off, av[1] + off, av[2] + off, av[3] + off);
            __syncwarp();
            if (lane == 0) mbar_arrive(&dready[s]);
            return true;
        };
        // two register sets in turn, so a load is first used a whole chunk after it was issued
        float r0[4] = {0.f, 0.f, 0.f, 0.f}, r1[4] = {0.f, 0.f, 0.f, 0.f};
        if (nc > 0) load_dt(0, r0);
        for (int c = 0; c < nc; c += 2) {
            if (!step(c, r0, r1)) break;
            if (c + 1 < nc && !step(c + 1, r1, r0)) break;
        }
        if (lane == 0) {
            // copies still in flight must land before the CTA may exit
            for (int u = (issued > 2 ? issued - 2 : 0); u < issued; u++) {
                mbar_wait(&full[u & 1], (u >> 1) & 1);
                mbar_wait(&fullx[u & 1], (u >> 1) & 1);
            }
        }
    } else if (warp == kEpiWarps + 1) {
        if (lane == 0) {
            constexpr uint32_t idG = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idY = idesc_bf16(128, 64, false, true);
            constexpr uint32_t idS = idesc_bf16(128, 64, true, true);
            const int ksN = a.nstate / 16;
            // descriptors built once; a K step adds a constant to the start-address field
            const uint64_t dWX = sw128_desc(smem_addr(smem + kOffWX), 8192, 1024);
            const uint64_t dH = sw128_desc(smem_addr(smem + kOffH), 8192, 1024);
            // stage 0's tiles; stage s is s * kStage bytes further
            const uint32_t st0 = smem_addr(smem);
            const uint64_t dC0 = sw128_desc(st0, 16, 1024);                   // C: K-major over states
            const uint64_t dB0 = sw128_desc(st0 + kTileBC, 16, 1024);         // B: K-major (G's B operand)
            const uint64_t dBt0 = sw128_desc(st0 + kTileBC, kAtom, 1024);     // B read state-major (S's A operand)
            const uint64_t dX0 = sw128_desc(st0 + 2 * kTileBC, 8192, 1024);   // x: MN-major rows of 64 columns
            auto stage_off = [](int s) { return (uint64_t)(s * (kStage >> 4)); };
            // G of chunk c into buffer c & 1 (whose previous contents became M before chunk c - 1's Y)
            auto issue_g = [&](int c) -> bool {
                const int s = c & 1;
                if (!mbar_wait(&full[s], (c >> 1) & 1)) return false;
                fence_after_sync();
#pragma unroll
                for (int k = 0; k < 8; k++)
                    if (k < ksN)
                        umma_bf16(tmem + kColG + s * 128, dC0 + stage_off(s) + kmajor_step(k, kAtom),
                                  dB0 + stage_off(s) + kmajor_step(k, kAtom), idG, k > 0 ? 1u : 0u);
                umma_commit(&gfull[s]);
                return true;
            };
            bool ok = nc == 0 || issue_g(0);
            for (int c = 0; ok && c < nc; c++) {
                // the next chunk's G goes first if its tiles have landed, else after this chunk's Y
                bool g_next = c + 1 < nc && mbar_test(&full[(c + 1) & 1], ((c + 1) >> 1) & 1);
                if (g_next && !(ok = issue_g(c + 1))) break;
                // the accumulators were read out and the entering state's copy written (phase c:
                // the epilogue arrives once after writing the initial state, then after each chunk)
                if (!(ok = mbar_wait(yempty, c & 1))) break;
                if (*(volatile int*)abort_flag) break;
                fence_after_sync();
                const int s = c & 1;
                // Yo = C H: A = C (K-major over states), B = H (MN-major: one row per state)
#pragma unroll
                for (int k = 0; k < 8; k++)
                    if (k < ksN)
                        umma_bf16(tmem + kColYo, dC0 + stage_off(s) + kmajor_step(k, kAtom), dH + mnmajor_step(k), idY,
                                  k > 0 ? 1u : 0u);
                // S = B^T (w o x): A = the B tile as an MN-major operand (64-state atoms 16 KB apart)
                if (!(ok = mbar_wait(wready, c & 1))) break;
                fence_after_sync();
#pragma unroll
                for (int k = 0; k < kQ / 16; k++)
                    umma_bf16(tmem + kColS, dBt0 + stage_off(s) + mnmajor_step(k), dWX + mnmajor_step(k), idS,
                              k > 0 ? 1u : 0u);
                umma_commit(&empty[s]);   // C and B of the stage are free once these have read them
                umma_commit(sfull);       // the state update may start before M x
                // Yd = M x: A = M from TMEM (K-major rows), B = x (MN-major rows of 64 columns)
                if (!(ok = mbar_wait(mready, c & 1))) break;
                if (!(ok = mbar_wait(&fullx[s], (c >> 1) & 1))) break;
                fence_after_sync();
#pragma unroll
                for (int k = 0; k < kQ / 16; k++)
                    umma_bf16_ta(tmem + kColYd, tmem + kColM + 8 * k, dX0 + stage_off(s) + mnmajor_step(k), idY,
                                 k > 0 ? 1u : 0u);
                umma_commit(yfull);
                umma_commit(&emptyx[s]);
                if (c + 1 < nc && !g_next && !(ok = issue_g(c + 1))) break;
            }
            if (!ok) record_timeout(a.status, abort_flag);
            // every MMA issued must have completed before TMEM is freed
            umma_commit(done);
            mbar_wait(done, 0);
        }
    } else if (warp == kEpiWarps + 2) {
        if (lane == 0) {
            // output stores: each chunk's staged tile leaves by bulk tensor stores (rows past the
            // sequence end are not written).  This thread issues no proxy fences, so no other
            // thread's fence waits for these stores.
            for (int c = 0; c < nc; c++) {
                if (!mbar_wait(ystaged, c & 1)) {
                    record_timeout(a.status, abort_flag);
                    break;
                }
                const unsigned char* Yt = smem + kOffM;
                tma_store_3d(&tmY, Yt, h * kP, c * kQ, b);
                if constexpr (sizeof(Tout) == 4) tma_store_3d(&tmY, Yt + kAtom, h * kP + 32, c * kQ, b);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                mbar_arrive(yfree);
            }
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        }
    } else {
        // epilogue warps 0-7: TMEM lane quadrant `quad` (chunk rows / states 32 quad ..), column half `hf`
        const int quad = warp & 3, hf = warp >> 2, row = quad * 32 + lane;
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        const float Al2 = __ldg(a.A + h) * kLog2e;
        const float Dv = a.D != nullptr ? __ldg(a.D + h) : 0.f;
        const float bias = a.dt_bias != nullptr ? __ldg(a.dt_bias + h) : 0.f;
        unsigned char* Mt = smem + kOffM;
        unsigned char* WXt = smem + kOffWX;
        unsigned char* Ht = smem + kOffH;
        // the state rows of this thread: state `row`, head-dimension columns 32 hf .. + 31
        float Hs[32];
        const size_t hoff = ((size_t)unit * a.nstate + row) * kP + 32 * hf;
#pragma unroll
        for (int p = 0; p < 32; p++) Hs[p] = (a.h0 != nullptr && row < a.nstate) ? a.h0[hoff + p] : 0.f;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; e++) v[e] = Hs[8 * q + e];
            *reinterpret_cast<uint4*>(swz(Ht, row, 4 * hf + q)) = pack8(v);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(yempty);
        for (int c = 0; c < nc; c++) {
            const int buf = c & 1;
            float* dlb = dl + buf * kQ;
            float* s2b = s2 + buf * kQ;
            // (a wait that runs out is caught by the uniform check before M is built)
            if (!mbar_wait(&dready[buf], (c >> 1) & 1)) record_timeout(a.status, abort_flag);
            const float si = s2b[row];
            const float slast = s2b[kQ - 1];
            // ---- column factors of the blocks below M's diagonal: cf_j = exp(s_e - s_j) Delta_j with
            // e the last step of j's 32-step block, so that for i in a later block
            // exp(s_i - s_j) Delta_j = exp(s_i - s_e) cf_j with both exponents <= 0
            // (read only while M is built, after the barrier in the check below)
            if (hf == 0) cf[row] = ex2_approx(s2b[32 * quad + 31] - si) * dlb[row];
            // ---- w o x, row j = `row`, columns 32 hf .. + 31, w_j = exp(s_last - s_j) Delta_j;
            // the same x values stay in registers for this thread's D x term
            uint32_t xw[16];
            {
                if (!mbar_wait(&fullx[buf], (c >> 1) & 1)) record_timeout(a.status, abort_flag);
                const unsigned char* Xt = smem + buf * kStage + 2 * kTileBC;
                const float wj = ex2_approx(slast - si) * dlb[row];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const uint4 xv = *reinterpret_cast<const uint4*>(swz(const_cast<unsigned char*>(Xt), row, 4 * hf + q));
                    xw[4 * q] = xv.x; xw[4 * q + 1] = xv.y; xw[4 * q + 2] = xv.z; xw[4 * q + 3] = xv.w;
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        v[2 * e] = wj * bf16lo(xw[4 * q + e]);
                        v[2 * e + 1] = wj * bf16hi(xw[4 * q + e]);
                    }
                    *reinterpret_cast<uint4*>(swz(WXt, row, 4 * hf + q)) = pack8(v);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(wready);
            // ---- M row `row`, 32-step column blocks cb = 2 hf, 2 hf + 1 (K atom hf of the A operand)
            // G of this chunk
            const bool gw = mbar_wait(&gfull[buf], (c >> 1) & 1);
            if (!gw) record_timeout(a.status, abort_flag);
            if (!epi_all(gw && *(volatile int*)abort_flag == 0)) break;
            fence_after_sync();
            // M row `row` into TMEM (the A operand of M x): 32-step column block cb as 16 columns
            // of bf16 pairs at kColM + 16 cb.  Chunk c - 1's M x finished reading them before
            // its outputs were released (yfull).  The two blocks are a loop, not unrolled: the
            // epilogue's code then fits the instruction cache far better (measured: 10% faster).
#pragma unroll 1
            for (int cc = 0; cc < 2; cc++) {
                const int cb = 2 * hf + cc;
                uint32_t mp[16];
                if (cb > quad) {
                    // above the diagonal: zero
#pragma unroll
                    for (int i = 0; i < 16; i++) mp[i] = 0u;
                } else {
                    uint32_t r[32];
                    tmem_ld32(tl + kColG + buf * 128 + 32 * cb, r);
                    if (cb < quad) {
                        // below the diagonal block: the factored decay
                        const float ri = ex2_approx(si - s2b[32 * cb + 31]);
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            const float4 f0 = *reinterpret_cast<const float4*>(cf + 32 * cb + 8 * q);
                            const float4 f1 = *reinterpret_cast<const float4*>(cf + 32 * cb + 8 * q + 4);
                            const float fj[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
                            for (int e = 0; e < 8; e += 2)
                                mp[4 * q + e / 2] = pack_bf16x2(__uint_as_float(r[8 * q + e]) * ri * fj[e],
                                                                __uint_as_float(r[8 * q + e + 1]) * ri * fj[e + 1]);
                        }
                    } else {
                        // the diagonal block: the decay per element, zero above the diagonal
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            float v[8];
#pragma unroll
                            for (int e = 0; e < 8; e++) {
                                const int j = 32 * cb + 8 * q + e;
                                const float m = __uint_as_float(r[8 * q + e]) * ex2_approx(si - s2b[j]) * dlb[j];
                                v[e] = j <= row ? m : 0.f;
                            }
#pragma unroll
                            for (int e = 0; e < 8; e += 2) mp[4 * q + e / 2] = pack_bf16x2(v[e], v[e + 1]);
                        }
                    }
                }
                tmem_st16(tl + kColM + 16 * cb, mp);
            }
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(mready);
            // ---- wait for Yd, S, Yo of this chunk
            // ---- the state update needs only S (and C H done reading the state copy): it runs
            // while M x is still on the tensor core
            const bool sw = mbar_wait(sfull, c & 1);
            if (!sw) record_timeout(a.status, abort_flag);
            if (!epi_all(sw && *(volatile int*)abort_flag == 0)) break;
            fence_after_sync();
            // state: H' = exp(s_last) H + S for state `row`; its bf16 copy is the next chunk's operand
            {
                uint32_t r[32];
                tmem_ld32(tl + kColS + 32 * hf, r);
                const float dec = ex2_approx(slast);
#pragma unroll
                for (int p = 0; p < 32; p++) Hs[p] = fmaf(dec, Hs[p], __uint_as_float(r[p]));
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) v[e] = Hs[8 * q + e];
                    *reinterpret_cast<uint4*>(swz(Ht, row, 4 * hf + q)) = pack8(v);
                }
            }
            // the state copy is visible to the tensor core before any global store is in flight
            // (the proxy fence would otherwise wait for those stores too)
            fence_async_smem();
            const bool yw = mbar_wait(yfull, c & 1);
            if (!yw) record_timeout(a.status, abort_flag);
            if (!epi_all(yw && *(volatile int*)abort_flag == 0)) break;
            fence_after_sync();
            // outputs: y = Yd + exp(s_i) Yo + D x for step t0 + row, columns 32 hf .. + 31
            float y[32];
            {
                uint32_t yd[32], yo[32];
                tmem_ld32(tl + kColYd + 32 * hf, yd);
                tmem_ld32(tl + kColYo + 32 * hf, yo);
                const float es = ex2_approx(si);
#pragma unroll
                for (int e = 0; e < 16; e++) {
                    y[2 * e] = fmaf(Dv, bf16lo(xw[e]), fmaf(es, __uint_as_float(yo[2 * e]), __uint_as_float(yd[2 * e])));
                    y[2 * e + 1] =
                        fmaf(Dv, bf16hi(xw[e]), fmaf(es, __uint_as_float(yo[2 * e + 1]), __uint_as_float(yd[2 * e + 1])));
                }
            }
            // TMEM read out: hand the accumulators back
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(yempty);
            // stage the 128 x 64 output tile (128-byte swizzled rows; fp32: two 32-column boxes)
            // once the previous chunk's tile has been read out of the staging buffer, and write
            // it with bulk tensor stores (rows past the sequence end are not written)
            {
                const bool fw = c == 0 || mbar_wait(yfree, (c - 1) & 1);
                if (!fw) record_timeout(a.status, abort_flag);
                if (!epi_all(fw && *(volatile int*)abort_flag == 0)) break;
                unsigned char* Yt = Mt;
                if constexpr (sizeof(Tout) == 2) {
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) v[e] = y[8 * q + e];
                        *reinterpret_cast<uint4*>(swz(Yt, row, 4 * hf + q)) = pack8(v);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 8; q++)
                        *reinterpret_cast<float4*>(swz(Yt + hf * kAtom, row, q)) =
                            make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(ystaged);
            }
        }
        if (a.final_state != nullptr && row < a.nstate && *(volatile int*)abort_flag == 0) {
#pragma unroll
            for (int q = 0; q < 8; q++)
                reinterpret_cast<float4*>(a.final_state + hoff)[q] =
                    make_float4(Hs[4 * q], Hs[4 * q + 1], Hs[4 * q + 2], Hs[4 * q + 3]);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == kEpiWarps + 1) {
        fence_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

template <typename Tout>
cudaError_t launch_typed(const CUtensorMap& tmC, const CUtensorMap& tmB, const CUtensorMap& tmX, const SsdArgs& a,
                         int64_t batch, int units, cudaStream_t st) {
    // y as (H P, L, batch): a box is 128 steps of one head's 64 columns (fp32: 32 columns)
    alignas(64) CUtensorMap tmY;
    const uint64_t HP = (uint64_t)a.H * kP, L = (uint64_t)a.L, es = sizeof(Tout);
    const uint64_t dims[3] = {HP, L, (uint64_t)batch};
    const uint64_t strides[2] = {HP * es, L * HP * es};
    const uint32_t box[3] = {(uint32_t)(128 / es), (uint32_t)kQ, 1};
    cudaError_t e = tc::encode_map(&tmY, a.out, 3, dims, strides, box, true, false, es == 4);
    if (e != cudaSuccess) return e;
    e = prepare_kernel<ssd_chunk_kernel<Tout>>(kSmem);
    if (e != cudaSuccess) return e;
    ssd_chunk_kernel<Tout><<<units, kThreads, kSmem, st>>>(tmC, tmB, tmX, tmY, a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ssd_fwd(const ssm_ssd_fwd_params* p, cudaStream_t st) {
    const size_t state_bytes = (size_t)p->batch * p->nheads * p->dstate * kP * sizeof(float);
    if (p->seqlen == 0) {
        // no steps: the final state is the initial one
        if (p->final_state == nullptr) return cudaSuccess;
        if (p->h0 != nullptr)
            return cudaMemcpyAsync(p->final_state, p->h0, state_bytes, cudaMemcpyDeviceToDevice, st);
        return cudaMemsetAsync(p->final_state, 0, state_bytes, st);
    }
    alignas(64) CUtensorMap tmC, tmB, tmX;
    cudaError_t e;
    {
        // B and C as (N, groups, L, batch): a box is 64 states of one group over 128 steps
        const uint64_t N = (uint64_t)p->dstate, G = (uint64_t)p->ngroups, L = (uint64_t)p->seqlen;
        const uint64_t dims[4] = {N, G, L, (uint64_t)p->batch};
        const uint64_t strides[3] = {N * 2, G * N * 2, L * G * N * 2};
        const uint32_t box[4] = {64, 1, (uint32_t)kQ, 1};
        if ((e = tc::encode_bf16_map(&tmC, p->C, 4, dims, strides, box, true, true)) != cudaSuccess) return e;
        if ((e = tc::encode_bf16_map(&tmB, p->B, 4, dims, strides, box, true, true)) != cudaSuccess) return e;
    }
    {
        // x as (H P, L, batch): a box is one head's 64 columns over 128 steps
        const uint64_t HP = (uint64_t)p->nheads * kP, L = (uint64_t)p->seqlen;
        const uint64_t dims[3] = {HP, L, (uint64_t)p->batch};
        const uint64_t strides[2] = {HP * 2, L * HP * 2};
        const uint32_t box[3] = {64, (uint32_t)kQ, 1};
        if ((e = tc::encode_bf16_map(&tmX, p->x, 3, dims, strides, box, true, false)) != cudaSuccess) return e;
    }
    SsdArgs a;
    a.L = (int)p->seqlen;
    a.H = (int)p->nheads;
    a.heads_per_group = (int)(p->nheads / p->ngroups);
    a.nstate = (int)p->dstate;
    a.nbox = p->dstate > 64 ? 2 : 1;
    a.nchunks = (int)ceil_div(p->seqlen, (int64_t)kQ);
    a.cb_bytes = (uint32_t)(2 * a.nbox * kAtom);
    a.dt = static_cast<const __nv_bfloat16*>(p->dt);
    a.A = p->A;
    a.D = p->D;
    a.dt_bias = p->dt_bias;
    a.h0 = p->h0;
    a.final_state = p->final_state;
    a.out = p->out;
    a.softplus = p->delta_softplus ? 1 : 0;
    if ((e = tc::device_status_word(&a.status)) != cudaSuccess) return e;
    const int units = (int)(p->batch * p->nheads);
    return p->out_dtype == SSM_BF16 ? launch_typed<__nv_bfloat16>(tmC, tmB, tmX, a, p->batch, units, st)
                                    : launch_typed<float>(tmC, tmB, tmX, a, p->batch, units, st);
}

}  // namespace ssm
