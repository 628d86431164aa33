// Host driver for the double-float arithmetic of the re-decision path
// (speculative_decoding_draft_04_gb300/csrc/spec_df.cuh compiled as plain C++).
// Commands on stdin, one per line; results on stdout:
//   exp <x>                    -> hi lo of e^x (x given as a double, split)
//   tab                        -> 64 lines: hi lo of 2^(j/64)
//   dot <n> <a_1..a_n> <w_1..w_n>  (floats given as hex bit patterns)
//                              -> hi lo of the compensated sum of a_i * w_i
//   mul <ah> <al> <bh> <bl>    -> hi lo of the double-float product
//   add <ah> <al> <bh> <bl>    -> hi lo of the double-float sum
//   rcp <t>                    -> hi lo of 1/t
//   log <zh> <zl>              -> log(zh + zl) as "<double> 0"
//   dot2 <n> <a..> <w..>       -> hi lo of the Dot2 dot product (hex floats)
//   div <ah> <al> <bh> <bl>    -> hi lo of the double-float quotient
//   sig <zh> <zl>              -> hi lo of 1 / (1 + e^{-(zh + zl)})
//   tanh <zh> <zl>             -> hi lo of tanh(zh + zl)
//   bf16 <hi hex> <lo hex>     -> "<bf16 bits> 0": nearest bfloat16 of hi + lo
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../speculative_decoding_draft_04_gb300/csrc/spec_df.cuh"

using spec::df;

static float from_bits(unsigned long x) {
  uint32_t u = (uint32_t)x;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}
static void put(df v) { std::printf("%.17g %.17g\n", (double)v.hi, (double)v.lo); }

int main() {
  df tab[spec::DD_EXP_TAB];
  for (int j = 0; j < spec::DD_EXP_TAB; ++j) spec::dd_exp_table_entry(tab, j);
  char cmd[16];
  while (std::scanf("%15s", cmd) == 1) {
    const std::string c(cmd);
    if (c == "exp") {
      double x;
      if (std::scanf("%lf", &x) != 1) return 1;
      put(spec::dd_exp(spec::dd_from_double(x), tab));
    } else if (c == "tab") {
      for (int j = 0; j < spec::DD_EXP_TAB; ++j) put(tab[j]);
    } else if (c == "dot" || c == "dot2") {
      int n;
      if (std::scanf("%d", &n) != 1) return 1;
      std::vector<float> a(n), w(n);
      for (int i = 0; i < n; ++i) {
        unsigned long x;
        if (std::scanf("%lx", &x) != 1) return 1;
        a[i] = from_bits(x);
      }
      for (int i = 0; i < n; ++i) {
        unsigned long x;
        if (std::scanf("%lx", &x) != 1) return 1;
        w[i] = from_bits(x);
      }
      if (c == "dot2") {
        spec::DdDot k;
        for (int i = 0; i < n; ++i) k.add(a[i], w[i]);
        put(k.value());
      } else {
        spec::DdSum k[4];
        for (int i = 0; i < n; ++i) k[i & 3].add(spec::rn_mul(a[i], w[i]));
        put(spec::dd_add(spec::dd_add(k[0].value(), k[1].value()), spec::dd_add(k[2].value(), k[3].value())));
      }
    } else if (c == "rcp") {
      float t;
      if (std::scanf("%f", &t) != 1) return 1;
      put(spec::dd_recip(t));
    } else if (c == "log") {
      float zh, zl;
      if (std::scanf("%f %f", &zh, &zl) != 2) return 1;
      std::printf("%.17g 0\n", spec::dd_log(df{zh, zl}, tab));
    } else if (c == "tanh") {
      float zh, zl;
      if (std::scanf("%f %f", &zh, &zl) != 2) return 1;
      put(spec::dd_tanh(df{zh, zl}, tab));
    } else if (c == "bf16") {
      unsigned long h, l;
      if (std::scanf("%lx %lx", &h, &l) != 2) return 1;
      std::printf("%u 0\n", (unsigned)spec::dd_to_bf16_bits(df{from_bits(h), from_bits(l)}));
    } else if (c == "sig") {
      float zh, zl;
      if (std::scanf("%f %f", &zh, &zl) != 2) return 1;
      put(spec::dd_sigmoid(df{zh, zl}, tab));
    } else if (c == "mul" || c == "add" || c == "div") {
      float ah, al, bh, bl;
      if (std::scanf("%f %f %f %f", &ah, &al, &bh, &bl) != 4) return 1;
      const df a = {ah, al}, b = {bh, bl};
      put(c == "mul" ? spec::dd_mul(a, b) : c == "add" ? spec::dd_add(a, b) : spec::dd_div(a, b));
    } else {
      return 2;
    }
  }
  return 0;
}
