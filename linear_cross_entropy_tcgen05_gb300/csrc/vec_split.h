/* vec_split.h -- split a run of elements into an unaligned head, a body of whole
 * 16-byte vectors and a tail, so that the body can be read with 16-byte vector loads.
 *
 * The TransformerEngine cross-entropy pull request (#995) describes this split for
 * rows of bf16 logits whose length (1025) is not a multiple of 8: row 0 is 1024
 * vector-aligned elements plus a 1-element tail, row 1 a 7-element head, 1016
 * aligned elements and a 2-element tail, row 2 a 6-element head, 1016 and a
 * 3-element tail. The library uses it for the targets and LSE arrays, whose base
 * pointers are only guaranteed 4-byte aligned.
 *
 * Plain C, usable from host and device code.
 */
#ifndef FLCE_VEC_SPLIT_H_
#define FLCE_VEC_SPLIT_H_

#include <stdint.h>

#if defined(__CUDACC__)
#define FLCE_HD __host__ __device__
#else
#define FLCE_HD
#endif

typedef struct {
  int64_t head; /* elements before the first 16-byte boundary */
  int64_t body; /* elements in whole 16-byte vectors */
  int64_t tail; /* elements after the last whole vector */
} flce_vec_split;

/* `start` is the element offset of the run from a 16-byte aligned address, `len`
 * its length in elements, `elem_bytes` the element size (a divisor of 16). */
static inline FLCE_HD flce_vec_split flce_split_for_vectors(int64_t start, int64_t len, int elem_bytes) {
  const int64_t per_vec = 16 / elem_bytes;
  const int64_t mis = start % per_vec;
  int64_t head = mis ? per_vec - mis : 0;
  if (head > len) head = len;
  const int64_t body = ((len - head) / per_vec) * per_vec;
  flce_vec_split s;
  s.head = head;
  s.body = body;
  s.tail = len - head - body;
  return s;
}

#endif /* FLCE_VEC_SPLIT_H_ */
