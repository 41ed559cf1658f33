// Host-side check of the double-float helpers the stochastic acceptance takes its decisions
// with (common.cuh: f2_add, f2_mul_f, f2_rcp, f2_gt), against exact fp64 arithmetic: a sum
// of two floats and a product of two floats are exact in fp64, so the double-float results
// must reproduce them exactly; the reciprocal must be within fp32 rounding of 1 / (hi + lo).
// Built and run by tests/test_f2_host.py; prints "ok <cases>" or the first failures.
#include <cmath>
#include <cstdint>
#include <cstdio>

#include "common.cuh"

using specv::F2;

static uint64_t state = 0x9E3779B97F4A7C15ull;
static uint64_t next_u64() {  // xorshift64*
  state ^= state >> 12;
  state ^= state << 25;
  state ^= state >> 27;
  return state * 0x2545F4914F6CDD1Dull;
}
static float rnd(float lo_exp, float hi_exp) {  // sign-random value with a log-uniform magnitude
  const double u = (double)(next_u64() >> 11) / 9007199254740992.0;
  const double e = lo_exp + (hi_exp - lo_exp) * u;
  const double m = std::ldexp(1.0, (int)std::floor(e)) * (1.0 + (double)(next_u64() >> 11) / 9007199254740992.0);
  return (float)((next_u64() & 1) ? m : -m);
}
static F2 norm(double x) {  // a normalised pair for x: hi = fp32(x), lo = fp32(x - hi)
  const float hi = (float)x;
  return F2{hi, (float)(x - (double)hi)};
}

int main() {
  int fails = 0, cases = 0;
  for (int t = 0; t < 200000; ++t) {
    const float a = rnd(-30.f, 30.f), b = rnd(-30.f, 30.f);
    // two floats: the sum and the product are exact in fp64
    const F2 s = specv::f2_add(F2{a, 0.f}, F2{b, 0.f});
    if ((double)s.hi + (double)s.lo != (double)a + (double)b && fails++ < 5)
      std::printf("add %a + %a -> %a %a\n", a, b, s.hi, s.lo);
    const F2 p = specv::f2_mul_f(F2{a, 0.f}, b);
    if ((double)p.hi + (double)p.lo != (double)a * (double)b && fails++ < 5)
      std::printf("mul %a * %a -> %a %a\n", a, b, p.hi, p.lo);
    // normalised pairs: the sum within 2^-44 of the operands' size, the order of fp64
    const double x = (double)rnd(-20.f, 20.f) * (1.0 + 1e-9 * (double)rnd(-1.f, 1.f));
    const double y = (double)rnd(-20.f, 20.f) * (1.0 + 1e-9 * (double)rnd(-1.f, 1.f));
    const F2 fx = norm(x), fy = norm(y);
    const double ex = (double)fx.hi + (double)fx.lo, ey = (double)fy.hi + (double)fy.lo;
    const F2 q = specv::f2_add(fx, fy);
    if (std::fabs((double)q.hi + (double)q.lo - (ex + ey)) > std::ldexp(std::fabs(ex) + std::fabs(ey), -44) &&
        fails++ < 5)
      std::printf("add2 %a %a + %a %a -> %a %a\n", fx.hi, fx.lo, fy.hi, fy.lo, q.hi, q.lo);
    if (specv::f2_gt(fx, fy) != (ex > ey) && fails++ < 5) std::printf("gt %a %a vs %a %a\n", fx.hi, fx.lo, fy.hi, fy.lo);
    // the reciprocal of a positive pair: within fp32 rounding (2^-23 relative)
    const F2 r_in = norm(std::fabs(x) + 1e-30);
    const double exact = 1.0 / ((double)r_in.hi + (double)r_in.lo);
    const float r = specv::f2_rcp(r_in);
    if (std::fabs((double)r - exact) > std::ldexp(exact, -23) && fails++ < 5)
      std::printf("rcp %a %a -> %a (exact %a)\n", r_in.hi, r_in.lo, r, exact);
    cases += 5;
  }
  if (specv::f2_rcp(F2{0.f, 0.f}) != 0.f || specv::f2_rcp(F2{-1.f, 0.f}) != 0.f) {
    std::printf("rcp of a non-positive input is not 0\n");
    ++fails;
  }
  if (fails) {
    std::printf("failures %d\n", fails);
    return 1;
  }
  std::printf("ok %d\n", cases);
  return 0;
}
