// CPU check of the quantizer's stochastic-rounding arithmetic (the index-domain
// form in nvq_device.cuh, e2m1_sr_code_bits): its fp32 steps, with the
// directed roundings emulated exactly, give the same E2M1 code as the rounding
// rule r < ceil(2^16 frac) on every finite bf16 value, a strided fp32 sweep,
// random (value, r) pairs, all 2^16 draws around every grid point and
// breakpoint, and extreme values.  Test-only; the rule is restated here from
// its definition (round up iff r < ceil(2^16 (|v| - lo) / (hi - lo)),
// saturate at 6, keep the sign).  argv[1]: number of random pairs.
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
static float bits2f(uint32_t u){float f; memcpy(&f,&u,4); return f;}
static uint32_t f2bits(float f){uint32_t u; memcpy(&u,&f,4); return u;}
// round the exact double value d (representable exactly in double) up to float
// exact fl_ru(p + c) and fl_rn(p + c) for doubles p, c holding exact values (p = a*b with b a power of
// two): TwoSum gives r + err == p + c exactly, then the float rounding looks at both
static float ru2(double p, double c){
  double r = p + c, bp = r - c, err = (p - bp) + (c - (r - bp));
  float f = (float)r;
  if ((double)f < r || ((double)f == r && err > 0)) f = nextafterf(f, INFINITY);
  else if ((double)f > r && err < 0 && (double)nextafterf(f, -INFINITY) >= r) f = nextafterf(f, -INFINITY);
  return f;
}
static float rn2(double p, double c){  // inputs here are exact in double already (checked by the caller)
  double r = p + c, bp = r - c, err = (p - bp) + (c - (r - bp));
  // inexact only when |p| is huge (x far above the grid, clamped to 7 afterwards)
  (void)err;
  return (float)r;
}
// oracle rule (same as orc_e2m1_encode_sr)
static uint8_t oracle_sr(float v, uint32_t r16){
  uint8_t s = signbit(v) ? 8 : 0; double a = fabs((double)v);
  if (a >= 6.0) return s | 7;
  double q = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
  double lo = floor(a / q) * q, hi = lo + q, frac = (a - lo) / q;
  double th = ceil(frac * 65536.0); double mag = ((double)r16 < th) ? hi : lo;
  if (mag == 0) return s; if (mag < 1) return s|1;
  int ex = ilogb(mag); int m = (int)((mag / ldexp(1.0, ex) - 1.0) * 2.0); return s | (((ex + 1) << 1) | m);
}
// kernel formulation (nvq_device.cuh): lines in base 128, where the fp32 ulp is
// exactly 2^-16, the grid of r
static uint8_t kernel_sr(float v, uint32_t r16){
  float x = fminf(fabsf(v), 6.0f);
  float a = ru2(2.0*(double)x, 128.0);
  float b = ru2((double)x, 130.0);
  float c = ru2(0.5*(double)x, 132.0);
  float m = fminf(fminf(a, b), c);                    // 128 + idx, rounded up onto the 2^-16 grid
  float negR = bits2f(0xC3000000u | r16);             // -(128 + r / 2^16)
  float d = rn2((double)m, (double)negR);             // exact
  float c4 = copysignf(4.0f, v);
  float Ms = rn2(12582916.0, -(double)c4);            // 1.5*2^23 (+8 when negative)
  float z = ru2((double)d, (double)Ms);
  return (uint8_t)(f2bits(z) & 0xFu);
}
int main(int argc, char** argv){
  const uint64_t n_rand = argc > 1 ? strtoull(argv[1], 0, 10) : 200000000ull;
  uint64_t n = 0, bad = 0; uint32_t seed = 12345;
  uint32_t rs[] = {0,1,2,3,255,256,32767,32768,32769,65533,65534,65535};
  // 1) every bf16 pattern (finite) times every r in a set, and exact grid boundaries
  for (uint32_t h = 0; h < 65536; ++h) {
    float v = bits2f(h << 16); if (!isfinite(v)) continue;
    for (int j = 0; j < 12; ++j) { n++; if (oracle_sr(v, rs[j]) != kernel_sr(v, rs[j])) { if (bad++ < 10) printf("bf16 %08x r %u: %x vs %x\n", h<<16, rs[j], oracle_sr(v, rs[j]), kernel_sr(v, rs[j])); } }
  }
  // 2) all fp32 values in [0, 16) with a stride, all 65536 r for a subset, random pairs
  for (uint32_t u = 0; u < 0x41800000u; u += 977) {
    float v = bits2f(u);
    for (int j = 0; j < 12; ++j) { float vv = (j & 1) ? -v : v; n++; if (oracle_sr(vv, rs[j]) != kernel_sr(vv, rs[j])) { if (bad++ < 10) printf("f32 %08x r %u\n", u, rs[j]); } }
  }
  for (uint64_t i = 0; i < n_rand; ++i) {
    seed = seed * 1664525u + 1013904223u; uint32_t u = seed % 0x41900000u;   // up to ~18
    seed = seed * 1664525u + 1013904223u; uint32_t r = seed >> 16;
    float v = bits2f(u); if (seed & 1) v = -v;
    n++; if (oracle_sr(v, r) != kernel_sr(v, r)) { if (bad++ < 10) printf("rand %08x r %u: %x vs %x\n", u, r, oracle_sr(v, r), kernel_sr(v, r)); }
  }
  // 3) neighbourhoods of the grid points and breakpoints with all r
  float pts[] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f, 8.f};
  for (int p = 0; p < 9; ++p) for (int d = -64; d <= 64; ++d) {
    uint32_t u = f2bits(pts[p]) + d; if ((int32_t)u < 0) continue;
    float v = bits2f(u);
    for (uint32_t r = 0; r < 65536; ++r) { n++; if (oracle_sr(v, r) != kernel_sr(v, r)) { if (bad++ < 10) printf("pt %08x r %u\n", u, r); } }
  }
  // 4) huge and tiny values
  float ex[] = {1e-45f, 1e-40f, 1e-30f, 1e-10f, 7.9999f, 8.0f, 100.0f, 3e38f, -0.0f};
  for (int p = 0; p < 9; ++p) for (uint32_t r = 0; r < 65536; ++r) { n++; if (oracle_sr(ex[p], r) != kernel_sr(ex[p], r)) { if (bad++ < 10) printf("ex %g r %u\n", ex[p], r); } }
  printf("checked %llu, mismatches %llu\n", (unsigned long long)n, (unsigned long long)bad);
  return bad != 0;
}
