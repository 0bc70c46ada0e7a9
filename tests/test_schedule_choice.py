"""The split-schedule choices of the D = 64 forward and the fused backward (host logic, no GPU).

The expected choices are the faster schedule measured back to back on GB300 (152 SMs) at each
shape; the library's cost models were fitted to those measurements and must keep choosing them.
"""
from __future__ import annotations

import pytest

import exact_attention_gb300 as fa

SMS = 152

# B, H, M, N, causal, split faster
FWD_CASES = [
    (1, 4, 2048, 2048, False, True),     # 18.8 against 24.3 us
    (1, 1, 8192, 8192, False, True),     # 31.6 against 80.5
    (1, 4, 4096, 4096, False, True),     # 28.9 against 43.1
    (4, 12, 2048, 2048, False, True),    # 60.5 against 65.1 (the headline workload)
    (4, 12, 1024, 1024, False, True),    # 22.8 against 26.0
    (1, 12, 512, 2048, False, True),     # 19.2 against 24.2
    (2, 12, 1024, 1024, False, False),   # whole 15.4 against 18.1
    (1, 16, 1024, 1024, False, False),   # whole 15.0 against 15.7
    (1, 8, 1024, 1024, False, False),    # whole 14.8 against 15.9
    (4, 12, 512, 512, False, False),     # even
    (16, 16, 4096, 4096, False, False),  # even (a part-empty last round of 27)
    (1, 4, 4096, 4096, True, True),      # causal, few pairs: 25.4 against 44.0
    (4, 12, 2048, 2048, True, False),    # causal: whole 44.1 against 50.9
    (4, 12, 1024, 1024, True, False),    # 17.2 against 26.3
    (1, 16, 8192, 8192, True, False),    # 151 against 167
    (1, 1, 1024, 1024, True, False),     # 14.9 against 34.8
]

BWD_CASES = [
    (1, 2, 1024, 1024, False),   # whole 21.7 against 23.1 us
    (1, 4, 2048, 2048, True),    # split 31.8 against 35.8
    (1, 8, 2048, 2048, False),   # whole 37.5 against 42.3
    (2, 12, 1024, 1024, True),   # split 39.3 against 41.1
    (4, 12, 1024, 1024, False),  # whole 59.0 against 61.5
    (4, 12, 2048, 2048, True),   # split 163.4 against 180.3 (the headline workload)
    (1, 1, 4096, 4096, True),    # split 34.3 against 58.9
    (1, 16, 1024, 1024, False),  # whole 25.2 against 31.4
    (1, 2, 8192, 8192, True),    # split 103.7 against 110.5
    (8, 16, 2048, 2048, False),  # whole 418 against 454
]


@pytest.mark.parametrize("B,H,M,N,causal,split", FWD_CASES)
def test_forward_split_choice(B, H, M, N, causal, split):
    assert fa.fa_debug_schedule_choice(0, B, H, M, N, causal, SMS) == int(split)


@pytest.mark.parametrize("B,H,M,N,split", BWD_CASES)
def test_backward_split_choice(B, H, M, N, split):
    assert fa.fa_debug_schedule_choice(1, B, H, M, N, False, SMS) == int(split)


def test_causal_backward_never_splits():
    assert fa.fa_debug_schedule_choice(1, 1, 1, 4096, 4096, True, SMS) == 0


def test_forced_schedules_and_invalid_queries():
    with fa.schedule(fa.FA_SCHED_FWD_SPLIT, 0):
        assert fa.fa_debug_schedule_choice(0, 4, 12, 2048, 2048, False, SMS) == 0
    with fa.schedule(fa.FA_SCHED_FWD_SPLIT, 1):
        assert fa.fa_debug_schedule_choice(0, 2, 12, 1024, 1024, False, SMS) == 1
    with fa.schedule(fa.FA_SCHED_BWD_SPLIT, 1):
        assert fa.fa_debug_schedule_choice(1, 8, 16, 2048, 2048, False, SMS) == 1
    assert fa.fa_debug_schedule_choice(0, 4, 12, 2048, 2048, False, SMS) == 1  # automatic again
    assert fa.fa_debug_schedule_choice(2, 1, 1, 128, 128, False, SMS) == -1
    assert fa.fa_debug_schedule_choice(0, 0, 1, 128, 128, False, SMS) == -1
    assert fa.fa_debug_schedule_choice(0, 1, 1, 128, 128, False, 0) == -1
    assert fa.fa_debug_schedule_choice(0, 1 << 16, 1 << 16, 128, 128, False, SMS) == -1  # B*H past int
