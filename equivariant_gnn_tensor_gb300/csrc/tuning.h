// Process-wide launch tuning set through tp_set_tuning (tests and sweeps).
// Every change bumps `gen`, which is part of the launch-plan cache key, so a
// plan is never reused across settings.
#pragma once
#include <cstdint>

#include "../../include/tpconv.h"

namespace tpc {

// Upper limits of the ring kernel's warps per block and pieces per warp.
constexpr int kRingMaxWarps = 8;
constexpr int kRingMaxPiecesPerWarp = 16;

struct TuningState {
    tp_tuning t;
    uint32_t gen;
};

TuningState tuning_snapshot();

}  // namespace tpc
