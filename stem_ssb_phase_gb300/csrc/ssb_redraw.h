// Host-side declarations of the redraw without the loss (ssb_redraw.cu).
#pragma once

#include "ssb_internal.h"

namespace ssb {

// BF slices of the spectral sum and the size of its slice buffer (double2).
int redraw_slices(int n_bf);
size_t redraw_part_elems(int N, int n_bf);
// Per-trial tables, then the spectral sum over the BF pixels and one 2-D inverse
// transform: a.Osum receives the unnormalised object accumulator [ry][rx] (as an
// evaluation with want_object leaves it); phase_out (arg O) and obj_out (O / (N^2 n_bf)),
// each [N][N], are written when not null.  part: redraw_part_elems; S, T: N x N complex64.
cudaError_t launch_redraw(const ObjectiveArgs &a, const ssb_params &theta, double2 *part, float2 *S,
                          float2 *T, float *phase_out, float2 *obj_out, cudaStream_t s);

}  // namespace ssb
