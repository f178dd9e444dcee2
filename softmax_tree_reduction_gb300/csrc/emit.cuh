// Writing one merged state of a thread block: the normalised result when the
// sequence is not split (P == 1), else the partial state for the combine.
#pragma once

#include "common.cuh"

namespace ta {

// o, l: merged numerator channel and denominator; M2: merged maximum in log2
// units (-inf for an empty slice).  `poison` marks a row whose length was
// invalid or whose block timed out: every value written is NaN.
__device__ __forceinline__ void emit_state(const SplitParams& p, int b, int hq, int split, int D,
                                           int dd, float o, float l, float M2, bool poison) {
    const size_t row = static_cast<size_t>(b) * p.Hq + hq;
    const float nan = __int_as_float(0x7fc00000);
    if (p.P == 1) {
        float ov, lv;
        if (poison) {
            ov = nan;
            lv = nan;
        } else if (l > 0.f) {
            ov = o / l;
            lv = (M2 + log2f(l)) * kLn2;
        } else {
            ov = 0.f;
            lv = -INFINITY;
        }
        if (in_bounds(row * D + dd, p.out_elems, p.err)) p.out[row * D + dd] = ov;
        if (dd == 0 && p.lse && in_bounds(row, p.rows, p.err)) p.lse[row] = lv;
    } else {
        const size_t pr = row * p.P + split;
        if (!in_bounds(pr, p.part_rows, p.err)) return;
        p.part_o[pr * D + dd] = poison ? nan : o;
        if (dd == 0) {
            p.part_m[pr] = poison ? nan : (M2 == -INFINITY ? -INFINITY : M2 * kLn2);
            p.part_l[pr] = poison ? nan : l;
        }
    }
}

}  // namespace ta
