"""The causal work order the host picks (``fattn_causal_order``; host only,
no GPU): heads per L2-sized group and whether units are handed out at run
time, against the rule written out here.

The rule: a group holds the K and V of as many heads as fit in 32 MiB
(2 * S * D * elem_bytes bytes a head); the heads are split into the fewest
such groups and the groups made near-equal (group size ceil(B*H / groups),
the kernel splitting the heads into groups of that size and one less); at
D = 128 groups are merged while one would hold fewer than 1.5 work units
(of 256 query rows) per SM.  D = 256 (CTA pairs) always takes units at run
time; D = 128 only when more than one group remains; D = 64 never."""
from __future__ import annotations

import math

import pytest

import exact_attention_forward_10_gb300 as fattn

SMS = 152


def expected(B, H, S, D, elem_bytes=2, sms=SMS):
    BH = B * H
    per_head = 2 * S * D * elem_bytes
    g = max(1, (32 << 20) // per_head)
    if g >= BH:
        groups = 1
    else:
        groups = math.ceil(BH / g)
        units = math.ceil(S / 256)
        while D == 128 and groups > 1 and math.ceil(BH / groups) * units < 3 * sms // 2:
            groups -= 1
    size = math.ceil(BH / groups)
    run_time = D == 256 or (D == 128 and size < BH)
    return {"group_heads": size if run_time else BH, "run_time": run_time}


@pytest.mark.parametrize("B,H,S,D,elem,group,run_time", [
    (2, 16, 8192, 128, 2, 8, True),    # 128 MiB of K, V: four groups of 8 heads
    (2, 16, 4096, 128, 2, 16, True),   # 64 MiB: two groups of 16
    (2, 16, 4097, 128, 2, 16, True),   # just over 64 MiB: 15+15+2 greedily; merged to 16+16
    (3, 11, 4096, 128, 2, 17, True),   # 33 heads: 11+11+11 hold 176 units < 228; 17+16
    (3, 12, 8192, 128, 2, 8, True),    # 36 heads: groups of 8 and 7 (the kernel's split)
    (1, 96, 2048, 128, 2, 32, True),   # 96 MiB: three groups of 32, 256 units each
    (2, 20, 4096, 128, 2, 20, True),   # 14+14+12 hold 224 units < 228: two of 20
    (1, 32, 2048, 128, 2, 32, False),  # 32 MiB: one group, static order
    (2, 16, 2048, 128, 2, 32, False),
    (2, 16, 16384, 128, 2, 4, True),
    (2, 16, 8192, 64, 2, 32, False),   # head dim 64: always static
    (2, 16, 8192, 256, 2, 4, True),    # CTA pairs: 32 MiB groups, always at run time
    (2, 16, 4097, 256, 2, 7, True),    # groups of 7 (the pair kernel: 7, 7, 7, 7, 4)
    (1, 4, 1024, 256, 2, 4, True),     # one group, still at run time on the pairs
    (2, 16, 8192, 128, 1, 16, True),   # E4M3: 64 MiB, two groups of 16
    (2, 16, 4096, 128, 1, 32, False),  # E4M3: 32 MiB, static
])
def test_orders_of_the_benchmark_shapes(B, H, S, D, elem, group, run_time):
    got = fattn.fattn_causal_order(B, H, S, D, elem, SMS)
    assert got == {"group_heads": group, "run_time": run_time}
    assert got == expected(B, H, S, D, elem)


def test_rule_over_many_shapes():
    for B in (1, 2, 3, 5):
        for H in (1, 3, 8, 11, 16, 24, 40):
            for S in (1, 255, 256, 1000, 2048, 4097, 8192, 12288, 20000):
                for D in (64, 128, 256):
                    got = fattn.fattn_causal_order(B, H, S, D, 2, SMS)
                    assert got == expected(B, H, S, D), (B, H, S, D, got)
                    g = got["group_heads"]
                    assert 1 <= g <= B * H
                    if not got["run_time"]:
                        assert g == B * H


@pytest.mark.parametrize("sms", [1, 16, 132, 152])
def test_merge_threshold_follows_the_sm_count(sms):
    for (B, H, S) in ((2, 16, 4097), (3, 11, 4096), (2, 20, 4096), (4, 8, 8192)):
        assert fattn.fattn_causal_order(B, H, S, 128, 2, sms) == expected(B, H, S, 128, 2, sms)


def test_errors():
    with pytest.raises(fattn.FattnError) as e:
        fattn.fattn_causal_order(2, 16, 4096, 128, 2, 0)
    assert e.value.status == fattn.FATTN_ERR_INVALID_ARG
    with pytest.raises(fattn.FattnError) as e:
        fattn.fattn_causal_order(2, 16, 4096, 128, 4, SMS)
    assert e.value.status == fattn.FATTN_ERR_INVALID_ARG
    with pytest.raises(fattn.FattnError) as e:
        fattn.fattn_causal_order(2, 16, 4096, 64, 1, SMS)
    assert e.value.status == fattn.FATTN_ERR_UNSUPPORTED
    with pytest.raises(fattn.FattnError) as e:
        fattn.fattn_causal_order(2, 16, 4096, 96, 2, SMS)
    assert e.value.status == fattn.FATTN_ERR_UNSUPPORTED
