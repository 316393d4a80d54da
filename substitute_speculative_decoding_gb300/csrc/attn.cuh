// Tree-masked GQA attention over the paged KV cache (see attn.cu).
#pragma once
#include <algorithm>
#include "common.cuh"

namespace sub {

struct AttnArgs {
  const uint16_t* Q;        // [n_q, Hq, D] bf16
  uint16_t* O;              // [n_q, Hq, D] bf16
  int n_q, n_heads_q, n_heads_kv, head_dim;
  // cache
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* page_table;
  int page_size, n_pages, layer;
  // key space
  int64_t n_prefix;             // committed keys [0, n_prefix) ...
  const int32_t* n_prefix_dev;  // ... or read on the device when non-null
  int64_t tree_base;            // position of tree slot 0 ...
  const int32_t* tree_base_dev; // ... or read on the device when non-null
  int n_slots;                  // tree slots [0, n_slots) addressable by this call
  const int32_t* anc;           // [n_q, anc_stride] root..self slot lists, or null (chain)
  int anc_stride;
  const int32_t* depth;         // [n_q] path length - 1 (with anc)
  int chain_slot0;              // chain mode: query i is slot chain_slot0 + i
  float scale;
  // 1: read the tree, the page table and the keys of other slots before the
  // launch wait (the model's decode path, whose predecessor is known to signal
  // its dependents only after its own wait); 0: every read after the wait
  int early_reads;
  // more key splits than one cluster holds (n_split = 8 C): each cluster's
  // merged partial goes to xpart [blocks][C][64][head_dim] with its row max
  // xm and denominator xl [blocks][C][64]; xcnt [blocks][8] counters start
  // at zero and are left at zero (attn_xpart_floats / attn_xcnt_count)
  float* xpart;
  float* xm;
  float* xl;
  unsigned int* xcnt;
};

constexpr int ATTN_MAX_SMEM = 200 * 1024;
// Key splits = CTAs of one thread-block cluster: up to 16 where the device
// runs 16-CTA clusters (a non-portable size), else the portable 8.
constexpr int ATTN_MAX_SPLIT = 16;
// Past one cluster, splits form clusters of 8 (more of them are co-resident
// than clusters of 16), merged across clusters through global scratch.
constexpr int ATTN_XCLUSTER = 8;
int32_t attn_init();
int attn_smem_bytes(const AttnArgs& a);
// Key splits for a launch; two_level allows 32 (two clusters, merged through
// the scratch above) when the caller can provide it.
int attn_pick_splits(const AttnArgs& a, int n_keys_hint, bool two_level = false);
size_t attn_xpart_floats(const AttnArgs& a, int n_split);   // xpart + xm + xl floats
size_t attn_xcnt_count(const AttnArgs& a, int n_split);
int32_t launch_tree_attn(const AttnArgs& a, int n_split, cudaStream_t st);

}  // namespace sub
