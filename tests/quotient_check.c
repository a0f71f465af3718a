/*
 * CPU check of the quantiser arithmetic used by the TMA-staged tile kernel
 * (test infrastructure; links the oracle's reference rounding).
 *
 * The kernel never divides.  For a group with maximum |x| = amax (a bf16
 * value) it forms
 *   s  = RN(RN(a/7) * 2^-6),  a = max(amax, 1e-12), RN(a/7) taken from
 *        y7 = RN(1/7) by one Markstein step: q0 = RN(a*y7), r = a - 7 q0,
 *        RN(q0 + r*y7)                         (claimed: s == RN(a/448))
 *   ny = an approximation of -1/s within one ulp (rcp.approx)
 * and for every x of the group (a bf16 value, |x| <= amax)
 *   q0 = RN(x*ny),  r = RN(s*q0 + x),  q1 = RN(r*ny + q0)  (= -x/s, nearly)
 *   code = e4m3(q1) with its sign bit flipped
 * (claimed: code == RNE_e4m3(clamp(RN(x/s), +-448)), the method's q, sign
 * of zero included).
 *
 * The program checks both claims for every bf16 amax (step `stride` through
 * the amax values, 1 = all of them), every bf16 x with |x| <= amax, both signs
 * of x, and each of the four floats nearest -1/s as ny: the two that bracket
 * it and their outer neighbours, so any approximation within one ulp is
 * covered.  Prints "tot=<cases> bad=<mismatches> scale_bad=<mismatches>".
 *
 * usage: quotient_check [stride]
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

uint8_t ora_e4m3_rne(float r);
float ora_group_scale(float amax);

static float from_bits(uint32_t u) {
  float x;
  memcpy(&x, &u, 4);
  return x;
}
static uint32_t to_bits(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  return u;
}

static float kernel_scale(float amax) {
  const float y7 = 1.0f / 7.0f;
  const float a = fmaxf(amax, 1e-12f);
  const float q0 = a * y7;
  const float r = fmaf(-7.0f, q0, a);
  return fmaf(r, y7, q0) * 0.015625f;
}

int main(int argc, char** argv) {
  const uint32_t stride = argc > 1 ? (uint32_t)strtoul(argv[1], NULL, 10) : 1u;
  unsigned long long tot = 0, bad = 0, scale_bad = 0;
  const long n_amax = (long)((0x7F80u + stride - 1) / stride);
#pragma omp parallel for schedule(dynamic, 16) reduction(+ : tot, bad, scale_bad)
  for (long ia = 0; ia < n_amax; ++ia) { /* every finite non-negative bf16 */
    const uint32_t ab = (uint32_t)ia * stride;
    const float amax = from_bits(ab << 16);
    const float s = ora_group_scale(amax);
    if (to_bits(kernel_scale(amax)) != to_bits(s)) scale_bad++;
    const double inv = -1.0 / (double)s;
    const float yr = (float)inv;
    const float ylo = (double)yr > inv ? nextafterf(yr, -INFINITY) : yr;
    const float yhi = (double)yr < inv ? nextafterf(yr, INFINITY) : yr;
    const float ny[4] = {nextafterf(ylo, -INFINITY), ylo, yhi, nextafterf(yhi, INFINITY)};
    for (uint32_t xb = 0; xb <= ab; ++xb) {
      for (int sg = 0; sg < 2; ++sg) {
        const float x = from_bits((xb << 16) | (sg ? 0x80000000u : 0u));
        const uint8_t ref = ora_e4m3_rne(x / s);
        for (int k = 0; k < 4; ++k) {
          const float q0 = x * ny[k];
          const float r = fmaf(s, q0, x);
          const float q1 = fmaf(r, ny[k], q0);
          if ((uint8_t)(ora_e4m3_rne(q1) ^ 0x80u) != ref) bad++;
        }
        tot++;
      }
    }
  }
  printf("tot=%llu bad=%llu scale_bad=%llu\n", tot, bad, scale_bad);
  return 0;
}
