// prefill_params.h -- argument block of the prefill kernels (host and device).
#pragma once

namespace tsa {

struct PrefillParams {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* states;    // [heads][DPAD*(dv+1)]
  float* scratch;   // [heads][n_spans][DPAD*(dv+1)], used when n_spans > 1
  long long N;
  int heads;
  int dv;
  int n_slices;
  int n_spans;
  int chunks_per_span;
  int accumulate;
};

}  // namespace tsa
