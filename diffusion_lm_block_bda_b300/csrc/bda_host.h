// bda_host.h -- host-side problem description shared by the planner and the
// C-ABI entry points.
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/bda_attn.h"

namespace bda {

struct Shape {
  int nseq = 0, hq = 0, hkv = 0, d = 0;
  int G = 1;        // hq / hkv
  int hg = 1;       // query heads packed into one 128-row tile
  int lg_hg = 0;
  int tok = 128;    // query tokens per tile = 128 / hg
  int kind = 0, B = 1;
  float scale = 0.f;
  int64_t total_q = 0, total_k = 0;
  int n_fwd = 0;    // forward work items (query tiles)
  int n_bwd = 0;    // backward work items (key tiles)
};

// Validates the problem and mask; fills `s`.  Host-only, launches nothing.
// A valid multi-block staircase gives BDA_ERR_UNSUPPORTED (no kernel takes it
// yet) unless count_only, for which it is BDA_OK.
bda_status validate(const bda_problem* p, const bda_mask_desc* m, Shape* s,
                    bool count_only = false);

size_t plan_bytes(const Shape& s);
size_t workspace_bytes(const Shape& s, bool with_bwd);
size_t ws_offset_D(const Shape& s);      // fp32 [hq][total_q]
size_t ws_offset_dqacc(const Shape& s);  // fp32 [total_q][hq][d]

// Writes the header and the LPT-ordered work items into `out` (plan_bytes).
void build_plan(const bda_problem* p, const bda_mask_desc* m, const Shape& s, uint8_t* out);

long long count_pairs(const bda_problem* p, const bda_mask_desc* m, const Shape& s);

// Records the text bda_last_cuda_error() returns on this thread.
void note_cuda_error(const char* text);

}  // namespace bda
