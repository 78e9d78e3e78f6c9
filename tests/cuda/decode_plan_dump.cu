// Prints the slice-per-SM decode GEMM's plan, as the library computes it, for
// shapes read from stdin ("M N K sms" per line): one line per shape,
//   ok R ctas groups kslices gparts warps nbox kbb wblk smem
// (ok = 0 and zeros where the kernel does not take the shape). Host code only:
// no GPU is needed to run it.
#include <cstdio>

#include "gemm_decode.cu"

int main() {
  long long M, N, K;
  int sms;
  while (std::scanf("%lld %lld %lld %d", &M, &N, &K, &sms) == 4) {
    const fp8blk::DecodePlan d = fp8blk::decode_plan(M, N, K, sms);
    if (!d.ok) {
      std::printf("0 0 0 0 0 0 0 0 0 0 0\n");
      continue;
    }
    std::printf("1 %d %d %d %d %d %d %d %d %d %zu\n", d.p.R, d.ctas, d.p.groups, d.p.kslices, d.p.gparts, d.warps,
                d.p.nbox, d.p.kbb, d.p.wblk, d.smem);
  }
  return 0;
}
