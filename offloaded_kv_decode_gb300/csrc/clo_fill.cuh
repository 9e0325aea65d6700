// clo_fill.cuh -- the miss-path fill's parameters and launch, shared by the
// stand-alone fill call and the layer call that carries the next layer's
// fill beside its attention ("CLO: CPU-Light KVCache Offloading", section 3
// Fig. 9: the next layer's missed heads move while the current layer
// computes).
#pragma once

#include "clo_device.cuh"

namespace clo {

constexpr int FILL_D = 128;  // head dimension (fp16 elements a row)

struct FillParams {
    const clo_half* srcK;
    const clo_half* srcV;
    const int32_t* tok;
    const int32_t* slot;  // nullptr: slot = token
    clo_half* cbK;
    clo_half* cbV;
    const int32_t* miss_list;
    const int32_t* miss_count;
    int32_t* err_flag;
    int T, k, C, n_heads;  // n_heads = B * Hkv
};

// Checks the arguments of a fill as clo_fill_cache_buffer documents them and
// fills p (sources as the device reads them).  Returns CLO_OK with
// nothing = true when there is nothing to move (B == 0 or k == 0).
clo_status make_fill_params(const clo_half* srcK, const clo_half* srcV, int T, const int32_t* tok,
                            const int32_t* slot, int k, clo_half* cbK, clo_half* cbV, int C,
                            const int32_t* miss_list, const int32_t* miss_count, int B, int Hkv,
                            int d, int32_t* err_flag, FillParams& p, bool& nothing);

// CTAs that keep every warp of a one-wave fill busy: one wave, and no more
// warps than 16-row steps of the longest possible miss list.
long long fill_max_grid(const FillParams& p);

// CTAs of a fill carried beside a kernel whose full grid is `wave` CTAs (that
// kernel then runs with this many fewer): a share of the wave, at least 1, at
// most fill_max_grid(p).
long long fill_beside_default_ctas(const FillParams& p, int wave);

// Launches the fill with `grid` CTAs on `stream`.
//  beside = false: the fill waits for the kernel before it (the lookup that
//    wrote the miss list) before it reads anything.
//  beside = true: for a fill launched directly after a libclo kernel that
//    writes nothing the fill reads or writes.  Such a kernel lets its
//    dependents start only once it has passed its own dependency wait, so
//    every kernel before it has finished: the fill reads the miss list at
//    once and runs beside that kernel on the SMs it leaves free, and waits
//    for it only at its end, so a kernel launched after the fill still
//    starts after both.
cudaError_t launch_fill(const FillParams& p, int grid, bool beside, cudaStream_t stream);

}  // namespace clo
