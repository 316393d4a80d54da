// Draft-tree expansion, target choice + accept walk, KV compaction.
#pragma once
#include "common.cuh"

namespace sub {

constexpr int MAX_WIDTH = 16;

struct ExpandArgs {
  const float* logits;   // [k_prev, V]
  int64_t V;
  float temp;
  sub_tree tree;
  int level;
  int k_prev;
  int n_chunks;
  // scratch: [k_prev * n_chunks * width] keys, [k_prev * n_chunks] max, sum; counter
  unsigned long long* part_key;
  float* part_max;
  float* part_sum;
  unsigned int* counter;   // zero before the first launch; the kernel leaves it zero
};
size_t expand_scratch_bytes(int k_prev, int n_chunks, int width);
int expand_pick_chunks(int k_prev, int64_t V);
int32_t launch_expand(const ExpandArgs& a, cudaStream_t st);

struct AcceptArgs {
  const float* logits;   // [n_nodes, V]
  int64_t V;
  sub_tree tree;
  int n_nodes;
  int mode;              // 0 greedy, 1 gumbel
  float temp;
  uint64_t seed;
  int64_t root_pos;
  const int32_t* root_pos_dev;   // overrides root_pos when non-null
  int n_chunks;
  unsigned long long* part_key;  // [n_nodes * n_chunks]
  unsigned int* counter;
  int32_t* accepted;     // [max_depth]
  int32_t* n_accepted;
  int32_t* bonus;
  int32_t* choice;       // [n_nodes] or null
  // emitted stream (model path only; null in the public entry point):
  // out_tokens[*state_emitted ...] += accepted tokens then the bonus
  int32_t* out_tokens;
  int32_t* state_emitted;
  int32_t* hist;         // accept histogram [max_depth + 1]
  // near-tie count (model path only; null in the public entry points): for
  // every node on the walked path, the runner-up's choice score per chunk goes
  // to part_key2 [n_nodes * n_chunks], and *near_ties counts the path nodes
  // whose best and runner-up choice scores differ by less than tie_gap
  unsigned long long* part_key2;
  int32_t* near_ties;
  float tie_gap;
  // adaptive depth: tree levels deeper than *depth_limit were not drafted
  // this cycle (their slots hold an earlier cycle's nodes); null = no limit
  const int32_t* depth_limit;
};
size_t accept_scratch_bytes(int n_nodes, int n_chunks);
int accept_pick_chunks(int n_nodes, int64_t V);
int32_t launch_accept(const AcceptArgs& a, cudaStream_t st);

struct CompactArgs {
  uint16_t* k;
  uint16_t* v;
  const int32_t* page_table;
  int n_layers, n_heads_kv, head_dim, page_size, n_pages;
  int64_t root_pos;
  const int32_t* root_pos_dev;    // overrides root_pos when non-null
  const int32_t* accepted;
  const int32_t* n_accepted;
  int max_accept;
};
int32_t launch_compact(const CompactArgs& a, cudaStream_t st);

}  // namespace sub
