/*
 * fa_seq_order.cuh -- longest-first order of the sequences of a paged batch.
 *
 * The forward kernel hands out work items statically (each CTA takes every
 * grid-th item, in a snake), so the order of the items decides the balance.
 * Paged decoding has one query token per sequence and key lengths that vary
 * by orders of magnitude; taking the sequences longest first (the longest-
 * processing-time-first rule) lets the short ones fill in behind the long
 * ones.  order[r] is the sequence of rank r: keys descending, ties by index
 * ascending, so the order is a deterministic permutation of 0..n-1.
 */
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace fa {

// The pre-pass is O(n^2) comparisons (n threads, each counting the sequences
// that rank before its own); past this many sequences the given order is used.
constexpr int64_t kMaxOrderedSeqs = 16384;

// order[r] for r < n from the key lengths seqused_k[0..n), each clamped to
// [0, cap] as the forward kernel clamps them.  One launch on `stream`.
cudaError_t launch_seq_order(const int32_t* seqused_k, int n, int64_t cap, int32_t* order,
                             cudaStream_t stream);

}  // namespace fa
