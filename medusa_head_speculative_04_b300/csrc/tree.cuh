// Device-resident tables of a fixed candidate tree (internal layout of medusa_tree).
#pragma once

#include <stdint.h>

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
};

struct medusa_tree {
  int32_t T = 0, P = 0, dmax = 0, mask_words = 0;
  int32_t max_rank[MEDUSA_MAX_DEPTH] = {};
  int device = 0;
  std::vector<int32_t> parent, depth, rank, child_start, child_count, paths, leaf;
  std::vector<uint32_t> mask;
  void* dev_block = nullptr;
  medusa_tree_dev dev{};
};
