/* Check of the quantize kernels' division by Q = 2^b - 1 (b = 2, 4, 8):
 *   q0 = RN(x * RN(1/Q)),  r = fma(-q0, Q, x),  q = fma(r, RN(1/Q), q0)
 * against the IEEE binary32 quotient RN(x / Q), for the finite x >= 0 whose
 * bit patterns are multiples of `stride` (stride 1: every one of them).
 * Prints the mismatch count per Q; exit status 1 if any.
 * Build: cc -O2 -ffp-contract=off -fno-fast-math -pthread divq_check.c -lm */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  uint32_t lo, hi, stride;
  float q, inv;
  uint64_t bad, checked;
} job_t;

static float from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static void *run(void *arg) {
  job_t *j = (job_t *)arg;
  uint32_t u = j->lo + (j->stride - j->lo % j->stride) % j->stride;
  for (; u < j->hi; u += j->stride) {
    const float x = from_bits(u);
    volatile float ref = x / j->q;
    const float q0 = x * j->inv;
    const float r = fmaf(-q0, j->q, x);
    const float q1 = fmaf(r, j->inv, q0);
    const float rv = ref;
    if (memcmp(&q1, &rv, 4) != 0) ++j->bad;
    ++j->checked;
    if (u > 0xFFFFFFFFu - j->stride) break;
  }
  return NULL;
}

int main(int argc, char **argv) {
  const uint32_t stride = argc > 1 ? (uint32_t)strtoul(argv[1], NULL, 10) : 1u;
  const float qs[3] = {3.0f, 15.0f, 255.0f};
  const float invs[3] = {0x1.555556p-2f, 0x1.111112p-4f, 0x1.010102p-8f};
  enum { kThreads = 8 };
  int failed = 0;
  for (int k = 0; k < 3; ++k) {
    if (1.0f / qs[k] != invs[k]) {
      printf("Q=%g: RN(1/Q) differs from the kernel constant\n", qs[k]);
      return 1;
    }
    pthread_t th[kThreads];
    job_t jb[kThreads];
    const uint64_t top = 0x7F800000u;   /* +inf excluded */
    for (int t = 0; t < kThreads; ++t) {
      jb[t] = (job_t){(uint32_t)(top * t / kThreads), (uint32_t)(top * (t + 1) / kThreads),
                      stride, qs[k], invs[k], 0, 0};
      pthread_create(&th[t], NULL, run, &jb[t]);
    }
    uint64_t bad = 0, checked = 0;
    for (int t = 0; t < kThreads; ++t) {
      pthread_join(th[t], NULL);
      bad += jb[t].bad;
      checked += jb[t].checked;
    }
    printf("Q=%g checked=%llu mismatches=%llu\n", qs[k], (unsigned long long)checked,
           (unsigned long long)bad);
    failed |= bad != 0;
  }
  return failed;
}
