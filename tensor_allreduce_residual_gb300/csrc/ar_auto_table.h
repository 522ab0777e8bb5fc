// ar_auto_table.h -- measured choices for AR_AUTO on the fused path
// (the heuristic_min_warp_number / selectImplementation analogue of
// "allreduce.d2").
//
// Each entry covers one (element size, R, packed units per row) shape and the
// token counts up to `tokens_max`; the first matching entry wins.  `strategy`
// is AR_ONESHOT (1) or AR_TWOSHOT (2); `vpt` is the packed vectors each
// thread of the one-shot kernel keeps per row (threads per row =
// units_row / vpt rounded up to a power of two).  Shapes with no entry fall
// back to the rule in ar_api.cu.
#pragma once

namespace ar {

struct AutoEntry {
    int esize;       // bytes per element
    int R;           // partials
    int units_row;   // 16-byte vectors per row
    int tokens_max;  // entry applies to tokens <= tokens_max
    int strategy;    // 1 = one-shot, 2 = two-shot
    int vpt;         // one-shot units per thread
};

// No measured entries yet: every shape takes the rule in ar_api.cu.
static const AutoEntry kAutoTable[] = {
    {0, 0, 0, 0, 0, 0},  // sentinel
};

}  // namespace ar
