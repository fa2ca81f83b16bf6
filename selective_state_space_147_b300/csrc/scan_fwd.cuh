// scan_fwd.cuh -- shared declarations of the selective-scan forward (see scan_fwd.cu).
#pragma once

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace ssm {

constexpr int kNMax = 16;     // state size handled per channel (padded)
constexpr int kTile = 64;     // time steps per B/C shared-memory tile
constexpr int kRow = 36;      // floats per staged time step: B[16] C[16] pad[4]
constexpr int kSub = 8;       // time steps per vector load

enum FwdMode { kFull = 0, kSummary = 1 };

struct FwdArgs {
    int64_t batch, dim, seqlen;
    int dstate;
    const void* u; const void* dt; const void* z; const void* B; const void* C; void* out;
    int64_t su_b, su_d, sdt_b, sdt_d, sz_b, sz_d, sB_b, sB_n, sC_b, sC_n, so_b, so_d;
    const float* A; const float* D; const float* bias; const float* h0;
    float* final_state; float* ckpt; int64_t ckpt_K, n_ckpt;
    int softplus;
    int vec_u, vec_dt, vec_z, vec_out, vec_BC;
    int64_t seg_len; int nseg;
    float* ws_hend;    // (channels, nseg, 16)
    float* ws_sdelta;  // (channels, nseg)
    float* ws_carry;   // (channels, nseg, 16)
    // one group of at most 16 states of a larger state: row strides of A and of
    // the (h0, final) states, checkpoint pairs in total and the group's first one
    int64_t sA, sst;
    int64_t ck_P, ck_p0;
    // B/C groups: channel d reads group d / cpg (group strides in elements)
    int64_t cpg, sB_g, sC_g;
};

template <typename Tin, typename Tout, bool ASYNC>
cudaError_t dispatch_G(const FwdArgs& a, int G, bool zoh, bool has_z, cudaStream_t st);

}  // namespace ssm
