"""The division by invariant integers the work-item decodes use (FastDiv in
attn_common.cuh; Granlund and Montgomery, "Division by invariant integers using
multiplication", 1994): with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
n / d = (umulhi(n, m) + n) >> l for every n < 2^31. Checked here against Python's
exact integer division for every divisor up to 4096 and large ones up to 2^31 - 1,
on the edges of each quotient step and on random n; the GPU parity tests exercise
the kernels' decodes over many (B, Hq, Hkv, T)."""
import random


def magic(d):
    l = 0
    while (1 << l) < d:
        l += 1
    m = ((1 << 32) * ((1 << l) - d)) // d + 1
    assert 0 < m < (1 << 32)
    return m, l


def fdiv(n, m, l):
    hi = (n * m) >> 32
    assert hi + n < (1 << 32)
    return (hi + n) >> l


def test_fastdiv_exact_for_all_n_below_2_31():
    rng = random.Random(5)
    top = (1 << 31) - 1
    divisors = list(range(1, 4097)) + [rng.randrange(4097, top) for _ in range(300)] + [top, (1 << 30) + 1, 65535,
                                                                                           1 << 20]
    for d in divisors:
        m, l = magic(d)
        ns = {0, 1, d - 1, d, d + 1, top, top - 1, (top // d) * d, (top // d) * d - 1}
        ns.update(rng.randrange(0, top + 1) for _ in range(200))
        ns.update(k * d + e for k in (1, 2, 7, 1000, top // d) for e in (-1, 0, 1) if 0 <= k * d + e <= top)
        for n in ns:
            assert fdiv(n, m, l) == n // d, (n, d)
