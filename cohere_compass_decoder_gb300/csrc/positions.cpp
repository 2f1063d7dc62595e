// Host helpers: MRoPE position ids of packed sequences and of decode tokens.
//
// Rule (mlxcel issue "Cohere Compass / North-Micro-Vision", section "Text decoder
// forward", paragraph "Position ids (get_rope_index)"): text tokens advance all three
// axes by one (a text token gets max(previous positions) + 1, the first token 0); the
// t*h*w tokens of an image get offset + (t_idx, h_idx, w_idx) over its merged grid in
// row-major order, offset = max(previous positions) + 1; the next text token continues
// at max + 1. rope_delta = max position + 1 - sequence length; a decode token sits at
// offset + rope_delta on all three axes.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "../../include/cc.h"

extern "C" cc_status cc_build_mrope_positions(const cc_image_span* spans, int32_t n_spans,
                                              const int32_t* seq_lens, int32_t n_seqs,
                                              int32_t* pos_out, int32_t* rope_delta_out) {
  if (n_seqs < 0 || n_spans < 0) return CC_ERR_INVALID_ARG;
  if (n_seqs > 0 && (!seq_lens || !rope_delta_out)) return CC_ERR_INVALID_ARG;
  if (n_spans > 0 && !spans) return CC_ERR_INVALID_ARG;
  int64_t total = 0;
  std::vector<int64_t> base(static_cast<size_t>(n_seqs) + 1, 0);
  for (int32_t s = 0; s < n_seqs; ++s) {
    if (seq_lens[s] < 0) return CC_ERR_INVALID_ARG;
    base[s] = total;
    total += seq_lens[s];
  }
  if (total > INT32_MAX) return CC_ERR_INVALID_ARG;
  if (total > 0 && !pos_out) return CC_ERR_INVALID_ARG;
  std::vector<std::vector<cc_image_span>> per(static_cast<size_t>(n_seqs));
  for (int32_t i = 0; i < n_spans; ++i) {
    const cc_image_span& sp = spans[i];
    if (sp.seq < 0 || sp.seq >= n_seqs || sp.start < 0 || sp.grid_t < 1 || sp.grid_h < 1 ||
        sp.grid_w < 1)
      return CC_ERR_INVALID_ARG;
    const int64_t n = static_cast<int64_t>(sp.grid_t) * sp.grid_h * sp.grid_w;
    if (static_cast<int64_t>(sp.start) + n > seq_lens[sp.seq]) return CC_ERR_INVALID_ARG;
    per[sp.seq].push_back(sp);
  }
  const int64_t T = total;
  for (int32_t s = 0; s < n_seqs; ++s) {
    auto& v = per[s];
    std::sort(v.begin(), v.end(),
              [](const cc_image_span& a, const cc_image_span& b) { return a.start < b.start; });
    int64_t next = 0;  // max(previous positions) + 1
    int64_t k = 0;     // token within the sequence
    const int64_t L = seq_lens[s];
    int32_t* pt = pos_out + base[s];
    int32_t* ph = pos_out + T + base[s];
    int32_t* pw = pos_out + 2 * T + base[s];
    for (const cc_image_span& sp : v) {
      if (sp.start < k) return CC_ERR_INVALID_ARG;  // overlapping images
      for (; k < sp.start; ++k) {
        pt[k] = ph[k] = pw[k] = static_cast<int32_t>(next);
        ++next;
      }
      const int64_t off = next;
      for (int32_t ti = 0; ti < sp.grid_t; ++ti)
        for (int32_t hi = 0; hi < sp.grid_h; ++hi)
          for (int32_t wi = 0; wi < sp.grid_w; ++wi, ++k) {
            pt[k] = static_cast<int32_t>(off + ti);
            ph[k] = static_cast<int32_t>(off + hi);
            pw[k] = static_cast<int32_t>(off + wi);
          }
      next = off + std::max({sp.grid_t, sp.grid_h, sp.grid_w});
      if (next > INT32_MAX) return CC_ERR_INVALID_ARG;
    }
    for (; k < L; ++k) {
      pt[k] = ph[k] = pw[k] = static_cast<int32_t>(next);
      ++next;
    }
    if (next > INT32_MAX) return CC_ERR_INVALID_ARG;
    rope_delta_out[s] = static_cast<int32_t>(next - L);
  }
  return CC_OK;
}

extern "C" cc_status cc_build_decode_positions(const int32_t* seq_lens, const int32_t* rope_delta,
                                               int32_t batch, int32_t* pos_out) {
  if (batch < 0) return CC_ERR_INVALID_ARG;
  if (batch == 0) return CC_OK;
  if (!seq_lens || !rope_delta || !pos_out) return CC_ERR_INVALID_ARG;
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t p = static_cast<int64_t>(seq_lens[b]) + rope_delta[b];
    if (seq_lens[b] < 0 || p < 0 || p > INT32_MAX) return CC_ERR_INVALID_ARG;
    pos_out[b] = pos_out[batch + b] = pos_out[2 * batch + b] = static_cast<int32_t>(p);
  }
  return CC_OK;
}
