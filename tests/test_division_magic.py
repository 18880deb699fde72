"""The multiply-high division the kernels use for a group's row within a unit
(div_small in the streaming kernels): with magic = floor(2^32 / d) + 1 the
high word of n * magic is floor(n / d) for every n with n * d < 2^32.  The
planner hands the kernels such a magic only when every n a unit can give
satisfies that (n < groups + units' groups), else 0 for a plain division.
These checks run the rule itself on the CPU: exhaustively for small
divisors, and at the edges of the allowed range for large ones."""
import random

import pytest


def _magic(d: int) -> int:
    return (1 << 32) // d + 1


def _div_small(n: int, magic: int) -> int:
    return (n * magic) >> 32


@pytest.mark.parametrize("d", list(range(2, 130)) + [192, 240, 480, 960, 1000, 4096, 8191])
def test_exact_over_the_allowed_range(d):
    m = _magic(d)
    assert m < (1 << 32)  # fits the 32-bit operand of the multiply-high
    limit = ((1 << 32) - 1) // d  # every n with n * d < 2^32
    rnd = random.Random(d)
    ns = set(range(0, min(limit, 5000) + 1))
    ns.update(rnd.randrange(0, limit + 1) for _ in range(2000))
    ns.update(range(max(0, limit - 2000), limit + 1))
    ns.update(k * d + r for k in (limit // d - 1, limit // d) for r in (-1, 0, 1) if 0 <= k * d + r <= limit)
    for n in ns:
        assert _div_small(n, m) == n // d, (n, d)


def test_the_planner_bound_is_needed():
    """Past n * d < 2^32 the rule can fail (here for a divisor whose magic
    carries the largest error), which is why the planner checks the bound."""
    d = 3
    m = _magic(d)
    bad = [n for n in range(((1 << 32) // d) - 10, ((1 << 32) // d) * 2, 12346)
           if _div_small(n, m) != n // d]
    assert bad, "expected the rule to fail somewhere beyond its bound"
