// Device-resident tables of a fixed candidate tree (internal layout of medusa_tree).
#pragma once

#include <stdint.h>

#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"

struct medusa_tree_dev {
  int32_t T, P, dmax, mask_words;
  const int32_t* parent;       // [T]
  const int32_t* depth;        // [T]
  const int32_t* rank;         // [T]
  const int32_t* child_start;  // [T] children of a node are contiguous in canonical order
  const int32_t* child_count;  // [T]
  const uint32_t* mask;        // [T * mask_words] ancestor-or-self bits
  const int32_t* paths;        // [P * (dmax+1)]
  const int32_t* leaf;         // [P]
  const int32_t* first_path;   // [T] lowest path index whose leaf descends from (or is) the node
};

struct medusa_tree {
  int32_t T = 0, P = 0, dmax = 0, mask_words = 0;
  int32_t max_rank[MEDUSA_MAX_DEPTH] = {};
  int device = 0;
  std::vector<int32_t> parent, depth, rank, child_start, child_count, paths, leaf, first_path;
  std::vector<uint32_t> mask;
  void* dev_block = nullptr;
  medusa_tree_dev dev{};
  // tree-tile visibility of query tiles, per (group size, rows per tile):
  // bit j of entry qt set iff a row of query tile qt may see a key of tree tile j
  std::mutex vis_mu;
  std::map<std::pair<int, int>, std::vector<uint64_t>> vis_cache;
};

// Visibility masks of the query tiles of a tree for group size G and rpt rows
// per tile (host; computed once per shape and cached in the tree).
const std::vector<uint64_t>& tree_tile_visibility(medusa_tree* t, int G, int rpt);
