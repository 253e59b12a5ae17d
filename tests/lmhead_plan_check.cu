// Host-only check of the fused LM head's launch plan, built by
// tests/test_launch_plans.py with nvcc (no GPU needed).  For every row-group
// size the host can choose (multiples of 64 up to kLmMaxRows), the plan
// functions of sv_lmhead.cuh must give:
//   - MMA shapes the two-CTA instruction accepts (N a multiple of 16, at most
//     256) and 32-column epilogue blocks;
//   - each CTA's half of an MMA's rows a whole number of 8-row swizzle atoms
//     and a legal TMA box;
//   - stage strides and operand offsets on 1024-byte boundaries;
//   - a ring of at least two stages inside the dynamic shared memory the
//     kernel opts into, with all of it below 2^18 bytes, where the
//     descriptors' start-address field would carry;
//   - accumulator slots that fit tensor memory and are reused by the tile
//     after next at the latest, which the two alternating tile-completion
//     barriers rely on;
//   - exactly one slot release per epilogue warp and slot use, with at most
//     three blocks of a slot per warp when the argmax epilogue loads them
//     together.
#include <cstdio>

#include "sv_lmhead.cuh"

int main() {
  int bad = 0, shapes = 0;
  // static shared memory of the kernel: two [4][kLmMaxRows] result arrays,
  // the draft tokens, barriers and scalars (a generous bound)
  const int kStatic = 2 * 4 * sv::kLmMaxRows * 4 + sv::kLmMaxRows * 4 + 512;
  const int kOptIn = 232448;  // bytes of shared memory a CTA may opt into
  for (int R = sv::kLmHBox; R <= sv::kLmMaxRows; R += sv::kLmHBox) {
    ++shapes;
    const int nmma = sv::lm_nmma(R), half = sv::lm_half_rows(R), nper = 2 * half;
    const int sb = sv::lm_stage_bytes(R), S = sv::lm_stages(sb);
    const int nslots = (sv::kLmTmemCols / nper < 2 * nmma) ? sv::kLmTmemCols / nper : 2 * nmma;
    const int nblk = nper / 32;
    int ok = 1;
    ok &= nmma >= 1 && nmma <= 2 && nmma * nper == R;
    ok &= nper % 32 == 0 && nper >= 32 && nper <= sv::kLmMaxN;
    ok &= half % 8 == 0 && half <= 256;
    ok &= sb % 1024 == 0 && (half * 128) % 1024 == 0 && sv::kLmABytes % 1024 == 0;
    ok &= sb == sv::kLmABytes + nmma * half * 128;
    ok &= S >= 2 && S <= sv::kLmMaxStages && S * sb <= sv::kLmRingBytes;
    ok &= sv::kLmRingBytes + 1024 + kStatic <= kOptIn;
    ok &= sv::kLmRingBytes + 1024 + kStatic < (1 << 18);
    ok &= nslots >= nmma && nslots <= sv::kLmMaxSlots && nslots * nper <= sv::kLmTmemCols;
    // slot reuse: the previous use of tile t's m-th slot is by tile t-1 or t-2
    for (int t = 0; t < 64; ++t)
      for (int m = 0; m < nmma; ++m) {
        const int g = t * nmma + m, prev = g - nslots;
        if (prev < 0) continue;
        const int pt = prev / nmma;
        ok &= pt >= t - 2 && pt <= t - 1;
      }
    // epilogue: warps of parity cb0 take blocks cb0, cb0 + 2, ...; each warp
    // releases a slot once (at cbl >= nblk - 2), after its last block of it
    for (int cb0 = 0; cb0 < 2; ++cb0)
      for (int m = 0; m < nmma; ++m) {
        int releases = 0, blocks = 0, last = -1;
        for (int cb = cb0; cb < R / 32; cb += 2) {
          if (cb / nblk != m) continue;
          ++blocks;
          last = cb - m * nblk;
          if (cb - m * nblk >= nblk - 2) ++releases;
        }
        ok &= releases == 1 && blocks >= 1 && last >= nblk - 2;
        if (nmma == 2) ok &= blocks <= 3;
      }
    if (!ok) {
      std::printf("bad plan: R=%d nmma=%d half=%d stage=%d stages=%d slots=%d\n", R, nmma, half,
                  sb, S, nslots);
      bad = 1;
    }
  }
  std::printf("%d row-group sizes checked\n", shapes);
  return bad;
}
