// Internal interface between the prefill GEMMs (fp9_prefill.cu) and the MoE
// prefill (fp9_moe_prefill.cu): the grouped launch, in which each token
// tile belongs to one FFN of a bank (a routed expert or a shared expert)
// and its rows to a contiguous range of a permuted activation buffer.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fp9moe.h"

namespace fp9 {

constexpr int kPrefillTileRows = 128;  // tokens per grouped tile

// Device table of a grouped launch, written by the MoE prefill's router:
// groups 0..n_routed-1 are the routed experts (FFN g of the routed bank),
// groups n_routed.. the shared experts. Group g owns rows
// [row[g], row[g] + cnt[g]) of the permuted buffers and m-tiles
// [mtile[g], mtile[g + 1]); mtile[n_groups] is the number of m-tiles.
struct GroupTableDev {
    const int32_t* row;    // [n_groups]
    const int32_t* cnt;    // [n_groups]
    const int32_t* mtile;  // [n_groups + 1]
    int32_t n_groups;
    int32_t n_routed;
};

// Both GEMMs of the grouped FFN: x16 [rows, H] fp16 -> h [rows, I] fp16
// (SwiGLU) -> y [rows, H] fp32 (unweighted per-row FFN outputs). With
// `split`, x16 and h hold two fp16 terms per value in the split layout
// ([rows, 2H] and [rows, 2I]: each 64-column chunk c as its hi terms in
// columns [128 c, 128 c + 64) and its lo terms in the next 64).
// max_mtiles bounds mtile[n_groups] (the launch grids are sized by it;
// CTAs past the real count exit at once).
fp9_status launch_grouped_ffn(const fp9_ffn_bank& routed, const fp9_ffn_bank* shared, const GroupTableDev& tab,
                              int64_t max_mtiles, const __half* x16, __half* h, float* y, int64_t rows, bool split,
                              int32_t* status, int sms, cudaStream_t stream);

}  // namespace fp9
