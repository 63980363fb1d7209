// Process-wide overrides of the library's measured kernel choices (tp_mlp_tuning.h). The
// launchers read them with one relaxed atomic load per knob: no environment lookup, no lock.
#include <atomic>

#include "internal.h"
#include "tp_mlp_tuning.h"

namespace tpk {
namespace {
std::atomic<int> g_tune[TP_TUNE_COUNT] = {
    {TP_TUNE_AUTO}, {TP_TUNE_AUTO}, {TP_TUNE_AUTO}, {TP_TUNE_AUTO},
    {TP_TUNE_AUTO}, {TP_TUNE_AUTO}, {TP_TUNE_AUTO}, {TP_TUNE_AUTO},
    {TP_TUNE_AUTO}, {TP_TUNE_AUTO}, {TP_TUNE_AUTO}, {TP_TUNE_AUTO}, {TP_TUNE_AUTO},
    {TP_TUNE_AUTO}, {TP_TUNE_AUTO}, {TP_TUNE_AUTO}, {TP_TUNE_AUTO}};
static_assert(TP_TUNE_COUNT == 17, "one initialiser per knob");
}  // namespace

int tuning(int knob) { return g_tune[knob].load(std::memory_order_relaxed); }

}  // namespace tpk

extern "C" {

tp_status tp_tuning_set(int32_t knob, int32_t value) {
  if (knob < 0 || knob >= TP_TUNE_COUNT) {
    tpk::set_last_error("unknown tuning knob");
    return TP_ERR_DTYPE;
  }
  if (value < TP_TUNE_AUTO) {
    tpk::set_last_error("tuning value below TP_TUNE_AUTO");
    return TP_ERR_SHAPE;
  }
  tpk::g_tune[knob].store(value, std::memory_order_relaxed);
  tpk::set_last_error("");
  return TP_OK;
}

int32_t tp_tuning_get(int32_t knob) {
  if (knob < 0 || knob >= TP_TUNE_COUNT) return TP_TUNE_AUTO - 1;
  return tpk::tuning(knob);
}

}  // extern "C"
