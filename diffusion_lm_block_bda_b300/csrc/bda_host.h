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
  int n_cgroups = 0;  // non-empty copy groups (multi-block staircase)
  // Split (decode) forward, for problems that fill few SMs: key tiles per
  // unit (0: no item is split), units, and partial-result slots.
  int split_c = 0;
  int n_dec = 0;
  int n_parts = 0;
};

// A problem with fewer than kSplitMaxUnits forward units (query tile x head
// group) fills under half of a B300's 148 SMs; its forward splits the key
// tiles of each query tile into chunks of split_c tiles, split_c chosen so
// the units number about kSplitTargetUnits.  Half the SMs with two key tiles
// each beat one tile on every SM for the decode step (14.3 against 16.4 us):
// each unit overlaps its second tile's loads with its first tile's work and
// writes half as many partial results.
constexpr int kSplitMaxUnits = 74;
constexpr int kSplitTargetUnits = 74;
// The backward's last wave, ordered longest-first: one dK/dV CTA per SM of a
// B300 (148 SMs).
constexpr int kTailWaveCtas = 148;

// Validates the problem and mask; fills `s`.  Host-only, launches nothing.
// A multi-block staircase whose non-empty groups are not in block order
// (visible decreasing along the sequence) is defined -- count_only accepts
// it -- but no kernel takes it: BDA_ERR_UNSUPPORTED.
bda_status validate(const bda_problem* p, const bda_mask_desc* m, Shape* s,
                    bool count_only = false);

// Plan bytes: header, forward items, (with_bwd) backward items, the
// copy-group table (int2 per non-empty group, padded to 16 bytes), then the
// split-forward units (DecItem each).
size_t plan_bytes(const Shape& s, bool with_bwd = true);
size_t plan_group_offset(const Shape& s, bool with_bwd);
size_t plan_dec_offset(const Shape& s, bool with_bwd);
// Workspace: the plan, then the split forward's partial results (fp32 O
// [n_parts * n_groups][d/4][128][4] and log2 LSE [n_parts * n_groups][128]).
size_t ws_offset_parts(const Shape& s);
size_t ws_offset_part_lse(const Shape& s);
size_t workspace_bytes(const Shape& s, bool with_bwd);
size_t ws_offset_D(const Shape& s);      // fp32 [hq][total_q]
size_t ws_offset_dqacc(const Shape& s);  // fp32 [total_q][hq][d]

// Writes the header and the LPT-ordered work items into `out`
// (plan_bytes(s, with_bwd) bytes; without the backward items, the header
// records n_bwd = 0).
void build_plan(const bda_problem* p, const bda_mask_desc* m, const Shape& s, uint8_t* out,
                bool with_bwd = true);

long long count_pairs(const bda_problem* p, const bda_mask_desc* m, const Shape& s);

// Records the text bda_last_cuda_error() returns on this thread.
void note_cuda_error(const char* text);

// TMA tensor maps over the caller's THD tensors (defined in bda_api.cu).
// bf16 [rows][heads][d]: box = 64 head-dim elements (128 bytes, 128B
// swizzle) x box_h heads x box_rows rows.
bool make_thd_map(void* map, const void* ptr, int d, int heads, int64_t rows, int box_h,
                  int box_rows);
// fp32 [rows][heads][d]: box = 32 floats (128 bytes, 128B swizzle) x box_h
// heads x box_rows rows.
bool make_f32_map(void* map, const void* ptr, int d, int heads, int64_t rows, int box_h,
                  int box_rows);
// e4m3 codes [rows][heads][d]: box = d codes x 1 head x 128 rows, no swizzle.
bool make_fp8_map(void* map, const void* ptr, int d, int heads, int64_t rows);

}  // namespace bda
