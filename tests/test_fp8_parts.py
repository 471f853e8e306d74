"""The error budget of the FP8 decode path's e4m3 operand parts, checked with
torch's own E4M3 conversion (round to nearest even), independent of the
kernels.

With an FP8 (E4M3) cache the decode products run on e4m3 tensor cores, so
the 16-bit query rows and the softmax weights enter as sums of e4m3 parts:
each query row is scaled by a power of two that puts its largest |q| in
[128, 256), part p is the E4M3 rounding of what parts 0..p-1 left, and the
weights enter as 256 P split into an E4M3 high part and the E4M3 rounding of
the remainder taken in fp16. These tests pin the claims the library makes
about that split: two parts hold a bf16 row exactly down to 2^-2 of the
scaled units, three parts hold an fp16 row to 12 significant bits, and two
parts hold 256 P to about 8 significant bits (for P >= 2^-10, and to 2^-18
absolute below). GPU parity of the FP8 path
against the fp64 oracle is in the gpu-marked tests.
"""
import math

import torch


def e4m3(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float8_e4m3fn).to(torch.float32)


def parts(row: torch.Tensor, n: int):
    """The row (fp32 values of 16-bit inputs) scaled by 2^e, then n parts."""
    mx = float(row.abs().max())
    e = 7 - math.floor(math.log2(mx)) if mx > 0 else 0
    v = row * (2.0 ** e)
    out = []
    for _ in range(n):
        p = e4m3(v)
        out.append(p)
        v = v - p
    return (2.0 ** e), out


def rows(dtype, seed, n=64, d=128):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, d, generator=g) * torch.exp(torch.randn(n, 1, generator=g) * 3)
    return x.to(dtype).to(torch.float32)


def test_two_parts_hold_a_bf16_row():
    for seed in range(4):
        for row in rows(torch.bfloat16, seed):
            s, (hi, lo) = parts(row, 2)
            scaled = row * s
            assert float(scaled.abs().max()) < 256 and float(hi.abs().max()) <= 256
            err = (scaled - (hi + lo)).abs()
            big = scaled.abs() >= 0.25
            assert not big.any() or float(err[big].max()) == 0.0
            # below 2^-2 the parts lose bits, by at most half a step of 2^-9
            assert float(err.max()) <= 2.0 ** -10


def test_three_parts_hold_an_fp16_row_to_12_bits():
    for seed in range(4):
        for row in rows(torch.float16, seed):
            s, (p0, p1, p2) = parts(row, 3)
            scaled = row * s
            err = (scaled - (p0 + p1 + p2)).abs()
            assert torch.all(err <= torch.maximum(scaled.abs() * 2.0 ** -12,
                                                  torch.full_like(err, 2.0 ** -10)))


def test_one_part_would_not_do():
    # a single e4m3 part is 4 significant bits: it misses the bf16 row by far
    row = rows(torch.bfloat16, 0)[0]
    s, (hi,) = parts(row, 1)
    assert float(((row * s) - hi).abs().max()) > 1.0


def test_two_parts_of_256p():
    g = torch.Generator().manual_seed(7)
    p = torch.exp2(-torch.rand(100000, generator=g) * 24)      # P in (2^-24, 1]
    x = 256.0 * p
    hi = e4m3(x)
    lo = e4m3((x.to(torch.float16) - hi.to(torch.float16)).to(torch.float32))
    err = (x - (hi + lo)).abs()
    # about 8 significant bits (4 + 4, plus the fp16 rounding of the
    # remainder) while the remainder part is a normal E4M3 value: P >= 2^-10
    big = x >= 2.0 ** -2
    rel = err[big] / x[big]
    assert float(rel.max()) <= 1.25 * 2.0 ** -8
    # below that the remainder part is subnormal: each smaller weight is off
    # by half an E4M3 step (2^-10) plus the remainder's fp16 rounding (at most
    # 2^-13 here), i.e. about 2^-18 of the largest weight 256
    assert float(err[~big].max()) <= 2.0 ** -10 + 2.0 ** -13
    assert float(hi.max()) <= 448.0
