// tuning.cu -- planner and dispatch overrides for measurement sweeps and
// tests (sgemm_set_tuning / sgemm_get_tuning).
//
// Every knob starts from its environment variable, read once while the
// library is loaded (a static initializer); the planner never calls getenv on
// the call path, so plans do not change with the process environment after
// load, and no getenv can race with a setenv in another thread.  Afterwards
// only sgemm_set_tuning changes a knob.  -1 means "the planner decides".
#include <atomic>
#include <cstdint>
#include <cstdlib>

#include "../../include/sgemm.h"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace {

struct KnobInfo {
    const char *env;
    int32_t lo, hi;   // accepted values besides -1
};

constexpr KnobInfo kKnobs[kKnobCount] = {
    {"SGEMM_FORCE_SPLIT", 1, kMaxSplit},
    {"SGEMM_FORCE_TAIL", 0, kMaxSplit},
    {"SGEMM_FORCE_TILE", 64, 128},
    {"SGEMM_FORCE_KERNEL", 0, 2},
    {"SGEMM_FORCE_TRANSPOSE_A", 0, 1},
    {"SGEMM_FFMA_EXT", 0, 1},
    {"SGEMM_TF32X3_FORCE_SPLIT", 1, 64},
    {"SGEMM_TF32X3_FORCE_TAIL", 0, 64},
    {"SGEMM_TF32X3_FUSE_A", 0, 1},
    {"SGEMM_WORKSPACE_LIMIT_MIB", 0, INT32_MAX},
    {"SGEMM_SCHEDULE", 0, 2},
    {"SGEMM_SK_MIN_SLICES", 1, 1 << 20},
    {"SGEMM_SK_GRID", 1, 1 << 20},
    {"SGEMM_TF32X3_BN", 128, 256},
};

bool valid(int k, int32_t v) {
    if (v == -1) return true;
    if (v < kKnobs[k].lo || v > kKnobs[k].hi) return false;
    if (k == kKnobTile) return v == 64 || v == 128;
    if (k == kKnobTf32x3Bn) return v == 128 || v == 256;
    return true;
}

std::atomic<int32_t> g_knobs[kKnobCount];

struct LoadEnv {
    LoadEnv() {
        for (int k = 0; k < kKnobCount; ++k) {
            int32_t v = -1;
            if (const char *s = std::getenv(kKnobs[k].env)) {
                char *end = nullptr;
                const long x = std::strtol(s, &end, 10);
                if (end != s && x >= INT32_MIN && x <= INT32_MAX && valid(k, int32_t(x)))
                    v = int32_t(x);
            }
            g_knobs[k].store(v, std::memory_order_relaxed);
        }
    }
};
const LoadEnv g_load_env;

}  // namespace

int32_t tuning(Knob k) { return g_knobs[k].load(std::memory_order_relaxed); }

}  // namespace sgemm_impl

extern "C" sgemm_status sgemm_set_tuning(int32_t knob, int32_t value) {
    using namespace sgemm_impl;
    if (knob < 0 || knob >= kKnobCount || !valid(knob, value)) return SGEMM_ERR_INVALID_ARG;
    g_knobs[knob].store(value, std::memory_order_relaxed);
    return SGEMM_OK;
}

extern "C" int32_t sgemm_get_tuning(int32_t knob) {
    using namespace sgemm_impl;
    if (knob < 0 || knob >= kKnobCount) return -2;
    return g_knobs[knob].load(std::memory_order_relaxed);
}
