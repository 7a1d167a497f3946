"""Segment length on the tensor-core path (host logic, checked on a real device: the rule
sizes itself by the device's SM count).

On dense rows, where the 16-chunk rule would apply, the library takes the segment length
of 8..64 chunks whose one-CTA-per-SM walks finish soonest: the (segment, head pair) items
in launch order (the segments of each row in turn, pairs fastest), each costing its chunk
count plus 2.5 chunk-times, handed to whichever SM is free first; the longest length within
1 % of the best wins.  The test restates that model in Python and reads the library's
choice back through the workspace size, which grows with the segment count and length.
Results do not depend on the segment length (the parity tests pin several); this only
checks which one is taken.
"""

import heapq

import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import state_space_model_ssd_gb300 as m
    from state_space_model_ssd_gb300 import build
    build.build()
    return m, torch.cuda.get_device_properties(0).multi_processor_count


def _makespan(row_chunks, rows, k, npairs, sms, c0=2.5):
    free = [0.0] * sms
    nseg = -(-row_chunks // k)
    for _ in range(rows):
        for s in range(nseg):
            ch = k if s + 1 < nseg else row_chunks - s * k
            for _ in range(npairs):
                heapq.heappush(free, heapq.heappop(free) + ch + c0)
    return max(free)


def _model_choice(row_chunks, rows, npairs, sms):
    spans = {k: _makespan(row_chunks, rows, k, npairs, sms) for k in range(8, 65)}
    best = min(spans.values())
    return max(k for k, v in spans.items() if v <= best * 1.01)


def _ws(m, torch, bsz, L, H, N, chunks=None, monkeypatch=None):
    if chunks is None:
        monkeypatch.delenv("SSD_SEGMENT_CHUNKS", raising=False)
    else:
        monkeypatch.setenv("SSD_SEGMENT_CHUNKS", str(chunks))
    x = torch.empty(bsz, L, H, 64, dtype=torch.bfloat16, device="meta")
    B = torch.empty(bsz, L, 1, N, dtype=torch.bfloat16, device="meta")
    return m.workspace_size(m.make_problem(x, B, -4.6), True)


@pytest.mark.parametrize("bsz,L,H,N", [
    (1, 32768, 80, 128),   # the mamba-2.8b layer at 32K tokens
    (2, 16384, 80, 128),   # two dense rows
    (1, 32768, 48, 128),
    (1, 65536, 24, 64),
    (1, 262144, 16, 64),   # genomics heads at 256K tokens
])
def test_segment_length_follows_the_makespan_model(env, monkeypatch, bsz, L, H, N):
    import torch
    m, sms = env
    k = _model_choice(L // 64, bsz, H // 2, sms)
    got = _ws(m, torch, bsz, L, H, N, monkeypatch=monkeypatch)
    assert got == _ws(m, torch, bsz, L, H, N, k, monkeypatch)
    assert got != _ws(m, torch, bsz, L, H, N, 16, monkeypatch) or k == 16


def test_segment_length_at_32k_is_46_chunks_on_152_sms(env, monkeypatch):
    import torch
    m, sms = env
    if sms != 152:
        pytest.skip("the figure is for a 152-SM device")
    assert _model_choice(512, 1, 40, sms) == 46
    assert _ws(m, torch, 1, 32768, 80, 128, monkeypatch=monkeypatch) == \
        _ws(m, torch, 1, 32768, 80, 128, 46, monkeypatch)


def test_other_problems_keep_the_default_rule(env, monkeypatch):
    """Packed sequences, small problems (under 16 chunks a segment by the default rule) and
    sequences of millions of tokens (64) are not sized by the model."""
    import torch
    m, _ = env
    # 2,097,152 tokens x 16 heads: 64-chunk segments
    assert _ws(m, torch, 1, 2097152, 16, 64, monkeypatch=monkeypatch) == \
        _ws(m, torch, 1, 2097152, 16, 64, 64, monkeypatch)
    # 2 x 2048 tokens x 24 heads: one-chunk segments fill the device
    assert _ws(m, torch, 2, 2048, 24, 128, monkeypatch=monkeypatch) == \
        _ws(m, torch, 2, 2048, 24, 128, 1, monkeypatch)
