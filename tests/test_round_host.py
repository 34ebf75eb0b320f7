"""SpecRound's call sequence on the host (no GPU): with the row pack, the first draft after each
selection writes it (or, with pack_in_select, the fused verify-select does), the other drafts read
it and the round's last draft drops it; without it, every draft is the plain call.  The binding's calls are replaced
by recorders, so only the sequencing is under test."""

import torch

from sparse_self_speculative_verify_gb300 import SpecRound
from sparse_self_speculative_verify_gb300 import binding as B


class _KV:
    """The attributes SpecRound reads from a KVCache, on the CPU."""
    device = torch.device("cpu")
    batch, h_kv, d, max_seq_len = 2, 2, 64, 128
    seq_lens = torch.tensor([100, 128], dtype=torch.int32)


def _record(monkeypatch):
    calls = []
    monkeypatch.setattr(B, "ssd_draft_pack_bytes", lambda kv, k_max: 4096)
    monkeypatch.setattr(B, "ssd_verify_attn", lambda *a, **k: calls.append("verify"))
    def verify_select(*a, pack=None, **k):
        assert pack is None or (pack.data_ptr() % 256 == 0 and pack.numel() == 4096)
        calls.append("verify_select" if pack is None else "verify_select+pack")
    monkeypatch.setattr(B, "ssd_verify_select", verify_select)
    monkeypatch.setattr(B, "ssd_select_topk", lambda *a, **k: calls.append("select"))
    monkeypatch.setattr(B, "ssd_draft_attn", lambda *a, **k: calls.append("draft"))

    def packed(kv, q, idx, cnt, scale, pack, mode, **k):
        assert pack.data_ptr() % 256 == 0 and pack.numel() == 4096
        calls.append({B.PACK_WRITE: "write", B.PACK_READ: "read", B.PACK_READ_DISCARD: "read+drop"}.get(mode, "?"))
    monkeypatch.setattr(B, "ssd_draft_attn_packed", packed)
    return calls


def _inputs(k=3):
    qv = torch.zeros((2, 3, 4, 64), dtype=torch.bfloat16)
    qd = torch.zeros((k, 2, 4, 64), dtype=torch.bfloat16)
    ks = torch.full((2,), 10, dtype=torch.int32)
    return qv, qd, ks


def test_pack_written_once_per_selection(monkeypatch):
    calls = _record(monkeypatch)
    r = SpecRound(_KV(), h_q=4, n_cand=3, k_max=70, workspace=B.Workspace())
    qv, qd, ks = _inputs()
    r.run(qv, qd, ks)
    assert calls == ["verify", "select", "write", "read", "read+drop"]  # the round's last draft drops it
    calls.clear()
    r.run(qv, qd, ks, fused_select=True)
    assert calls == ["verify_select", "write", "read", "read+drop"]
    calls.clear()
    r.draft(qd[0])  # another draft after the round: the pack was dropped, so it is written again
    r.draft(qd[0])  # and read by the next one
    r.select(ks)
    r.draft(qd[0])  # a new selection is written first
    assert calls == ["write", "read", "select", "write"]


def test_pack_written_by_the_select_when_asked(monkeypatch):
    calls = _record(monkeypatch)
    r = SpecRound(_KV(), h_q=4, n_cand=3, k_max=70, workspace=B.Workspace(), pack_in_select=True)
    qv, qd, ks = _inputs()
    r.run(qv, qd, ks, fused_select=True)
    assert calls == ["verify_select+pack", "read", "read", "read+drop"]
    calls.clear()
    r.run(qv, qd, ks)  # a separate select: the first draft writes the pack
    assert calls == ["verify", "select", "write", "read", "read+drop"]


def test_without_pack_every_draft_is_plain(monkeypatch):
    calls = _record(monkeypatch)
    r = SpecRound(_KV(), h_q=4, n_cand=3, k_max=70, workspace=B.Workspace(), pack_rows=False)
    qv, qd, ks = _inputs()
    r.run(qv, qd, ks)
    assert calls == ["verify", "select", "draft", "draft", "draft"]
    assert r.pack is None
