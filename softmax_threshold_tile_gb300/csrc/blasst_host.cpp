// Host-side controls that turn user settings into the kernel's threshold_scale_factor
// ("Skip-Softmax" design doc, vLLM-Omni: sections "From configuration to the kernel
// threshold", "Timestep gating" and "Mapping the cutoff to denoising steps"). No CUDA.

#include <cmath>
#include <cstdint>

#include "blasst.h"

extern "C" blasst_status blasst_factor_from_threshold(double threshold, int64_t max_kv_len,
                                                      double* factor) {
  // The direct control: the kernel divides the factor by max_kv_len, so passing
  // threshold * max_kv_len makes lambda equal to the threshold at any length.
  if (!factor || !std::isfinite(threshold) || threshold < 0.0 || max_kv_len < 1)
    return BLASST_ERR_INVALID_ARG;
  const double f = threshold * static_cast<double>(max_kv_len);
  if (!std::isfinite(f)) return BLASST_ERR_INVALID_ARG;
  *factor = f;
  return BLASST_OK;
}

extern "C" blasst_status blasst_factor_from_target_sparsity(double a, double b, double target_sparsity,
                                                            double* factor) {
  // The calibrated control: a point on the curve a * exp(b * s) fitted per model.
  if (!factor || !std::isfinite(a) || !std::isfinite(b) || !std::isfinite(target_sparsity))
    return BLASST_ERR_INVALID_ARG;
  const double f = a * std::exp(b * target_sparsity);
  if (!std::isfinite(f) || f < 0.0) return BLASST_ERR_INVALID_ARG;
  *factor = f;
  return BLASST_OK;
}

extern "C" blasst_status blasst_gate_factor(double factor, double disabled_until_timestep,
                                            int t_published, double t, double* out, int* warn) {
  if (!out || !std::isfinite(factor) || factor < 0.0 || !std::isfinite(disabled_until_timestep) ||
      disabled_until_timestep < 0.0)
    return BLASST_ERR_INVALID_ARG;
  if (warn) *warn = 0;
  if (disabled_until_timestep == 0.0) {  // sentinel: the gate is off and t is never read
    *out = factor;
    return BLASST_OK;
  }
  if (!t_published) {  // stay dense rather than guess from the step index
    if (warn) *warn = 1;
    *out = 0.0;
    return BLASST_OK;
  }
  if (!std::isfinite(t)) return BLASST_ERR_INVALID_ARG;
  *out = t > disabled_until_timestep ? 0.0 : factor;
  return BLASST_OK;
}

extern "C" blasst_status blasst_dense_steps(const double* t, int n, double disabled_until_timestep,
                                            int* dense_steps) {
  if (!dense_steps || n < 0 || (n > 0 && !t) || !std::isfinite(disabled_until_timestep))
    return BLASST_ERR_INVALID_ARG;
  int count = 0;
  for (int i = 0; i < n; ++i)
    if (t[i] > disabled_until_timestep) ++count;
  *dense_steps = count;
  return BLASST_OK;
}

extern "C" blasst_status blasst_flow_shift_schedule(double shift, int num_points, double* t_out) {
  if (!t_out || !std::isfinite(shift) || !(shift > 0.0) || num_points < 2) return BLASST_ERR_INVALID_ARG;
  for (int i = 0; i < num_points; ++i) {
    const double u = 1.0 - static_cast<double>(i) / static_cast<double>(num_points - 1);
    t_out[i] = shift * u / (1.0 + (shift - 1.0) * u);
  }
  return BLASST_OK;
}
