"""The block verification's integer division (csrc/exact_div.cuh) gives the
correctly rounded IEEE double quotient e / S for 1 <= e <= S < 2^50: the same
source compiled for the host, compared bit for bit with the hardware double
division on edge cases and ten million random pairs (no GPU)."""
import os
import subprocess
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "mla_block_diffusion_gb300", "csrc", "exact_div.cuh")

PROG = r"""
#include <stdio.h>
#include <string.h>
#include "exact_div.cuh"
using namespace ds;
static unsigned long long s_state = 0x9E3779B97F4A7C15ull;
static unsigned long long rnd() {  // splitmix64
    unsigned long long z = (s_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
static int check(unsigned long long e, unsigned long long S) {
    const ExactDivisor d = exact_divisor(S);
    const double got = exact_div(e, d), want = (double)e / (double)S;
    unsigned long long a, b;
    memcpy(&a, &got, 8);
    memcpy(&b, &want, 8);
    if (a != b) {
        printf("mismatch e=%llu S=%llu got=%.17g want=%.17g\n", e, S, got, want);
        return 1;
    }
    return 0;
}
int main(void) {
    int bad = 0;
    const unsigned long long top = (1ull << 50) - 1;
    unsigned long long edges[] = {1, 2, 3, 5, 7, 1ull << 20, (1ull << 32), (1ull << 32) + 1, (1ull << 33) - 1,
                                  (1ull << 49), top - 1, top};
    for (unsigned i = 0; i < sizeof(edges) / 8; ++i)
        for (unsigned j = 0; j < sizeof(edges) / 8; ++j) {
            const unsigned long long e = edges[i] < (1ull << 32) + 1 ? edges[i] : (1ull << 32), S = edges[j];
            if (e >= 1 && e <= S) bad += check(e, S);
        }
    for (int k = 0; k < 10000000 && bad < 10; ++k) {
        const int bitsS = 1 + (int)(rnd() % 50);
        unsigned long long S = (rnd() >> (64 - bitsS)) | 1ull;
        if (S > top) S = top;
        unsigned long long e;
        const unsigned long long emax = S < (1ull << 32) ? S : (1ull << 32);
        switch (k & 3) {
            case 0: e = 1 + rnd() % emax; break;
            case 1: e = emax; break;
            case 2: e = 1 + (rnd() >> (63 - (int)(rnd() % 33))) % emax; break;
            default: e = emax > 1 ? emax - 1 : 1;
        }
        bad += check(e, S);
    }
    // powers of two and near-ties: S = 2^k * odd small, e chosen to land exactly halfway
    for (int k = 0; k < 50; ++k)
        for (unsigned long long m = 1; m < 64; m += 2) {
            const unsigned long long S = m << k;
            if (S > top) break;
            for (unsigned long long e = 1; e <= 64 && e <= S; ++e) bad += check(e, S);
        }
    printf(bad ? "FAIL\n" : "ok\n");
    return bad != 0;
}
"""


def test_exact_division_matches_ieee():
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "t.cpp"), os.path.join(d, "t")
        open(src, "w").write(PROG)
        subprocess.run(["g++", "-O2", "-std=c++17", "-I", os.path.dirname(HDR), src, "-o", exe], check=True)
        r = subprocess.run([exe], capture_output=True, text=True)
        assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:]
