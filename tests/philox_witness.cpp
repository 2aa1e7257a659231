// Library witness for the oracle's Philox4x32-10: PyTorch's own counter-based engine
// (ATen/core/PhiloxRNGEngine.h), driven through its public constructor.
// philox_engine(seed, subsequence, offset) keys the generator with the 64-bit seed and
// starts at counter (offset low, offset high, subsequence low, subsequence high); its
// first four outputs are the four words of that counter's block.
// Reads lines "seed subsequence offset" on stdin, prints the four words in hex.
#include <ATen/core/PhiloxRNGEngine.h>
#include <cinttypes>
#include <cstdio>

int main() {
  unsigned long long seed, sub, off;
  while (std::scanf("%llu %llu %llu", &seed, &sub, &off) == 3) {
    at::philox_engine e(seed, sub, off);
    uint32_t w0 = e(), w1 = e(), w2 = e(), w3 = e();
    std::printf("%08" PRIx32 " %08" PRIx32 " %08" PRIx32 " %08" PRIx32 "\n", w0, w1, w2, w3);
  }
  return 0;
}
