"""B and C shared by groups of heads, on the CPU oracle.

A group of H/G consecutive heads reads one B and one C per token (head h
reads group h // (H/G)).  Sharing is only an addressing change, so
running the oracle on grouped B/C must give exactly the results of the
per-head layout with each group's B/C copied to its heads.  Any other
head-to-group map (h % G, the group count swapped with the group size)
gives another result for the shapes below, where G is neither 1 nor H.
"""
import numpy as np
import pytest

import oracle
import synth


def _expand(a, H):
    """Per-head copy of a grouped B/C tensor (groups on axis 2)."""
    return np.repeat(a, H // a.shape[2], axis=2)


@pytest.mark.parametrize("G", [1, 2, 4])
@pytest.mark.parametrize("R", [1, 2])
def test_prefill_grouped_equals_per_head_copy(G, R):
    wl = synth.Workload("t", "prefill", 2, 37, 4, 8, 16, R, "bf16", chunk=16, h0_std=0.2, carry=True,
                        ngroups=G)
    inp = synth.prefill_inputs(wl)
    assert inp["B"].shape == (2, 37, G, R, 16)
    kw = dict(batch=2, L=37, H=4, P=8, N=16, R=R, dtype="bf16", h0=inp["h0"], prev_B=inp["prev_B"],
              prev_x=inp["prev_x"], nthreads=1)
    y, h, pB, px, _ = oracle.prefill(inp, **kw)
    per_head = dict(inp, B=_expand(inp["B"], 4), C=_expand(inp["C"], 4))
    y2, h2, pB2, px2, _ = oracle.prefill(per_head, **kw)
    assert np.array_equal(y, y2)
    assert np.array_equal(h, h2)
    assert np.array_equal(pB, pB2)  # the carry is the unit's last B, i.e. its group's
    assert np.array_equal(px, px2)


def test_prefill_grouped_wrong_map_differs():
    """The head-to-group map is not invisible: mapping head h to group
    h % G instead changes the outputs of heads 1 and 2 (H 4, G 2)."""
    wl = synth.Workload("t", "prefill", 1, 20, 4, 8, 16, 1, "bf16", chunk=16, ngroups=2)
    inp = synth.prefill_inputs(wl)
    kw = dict(batch=1, L=20, H=4, P=8, N=16, R=1, dtype="bf16", nthreads=1)
    y, _, _, _, _ = oracle.prefill(inp, **kw)
    wrong = {k: v for k, v in inp.items()}
    for k in ("B", "C"):
        wrong[k] = inp[k][:, :, [0, 1, 0, 1]]  # per head: group h % 2
    y2, _, _, _, _ = oracle.prefill(wrong, **kw)
    assert np.array_equal(y[:, :, [0, 3]], y2[:, :, [0, 3]])
    assert not np.allclose(y[:, :, [1, 2]], y2[:, :, [1, 2]])


def test_prefill_grouped_varlen_equals_per_head_copy():
    wl = synth.Workload("t", "varlen", 1, 0, 4, 8, 16, 1, "bf16", chunk=16, nseq=3, len_lo=3, len_hi=30,
                        ngroups=2)
    lens = synth.lengths(3, 3, 30, seed=0)
    wl.cu_seqlens = synth.varlen_cu_seqlens(lens)
    wl.seqlen = int(wl.cu_seqlens[-1])
    inp = synth.prefill_inputs(wl)
    kw = dict(batch=1, L=wl.seqlen, H=4, P=8, N=16, R=1, dtype="bf16", cu_seqlens=wl.cu_seqlens, nthreads=1)
    y, h, _, _, _ = oracle.prefill(inp, **kw)
    y2, h2, _, _, _ = oracle.prefill(dict(inp, B=_expand(inp["B"], 4), C=_expand(inp["C"], 4)), **kw)
    assert np.array_equal(y, y2)
    assert np.array_equal(h, h2)


@pytest.mark.parametrize("G", [1, 2])
def test_decode_grouped_equals_per_head_copy(G):
    wl = synth.Workload("t", "decode", 3, 0, 4, 8, 16, 2, "bf16", h0_std=0.1, carry=True, ngroups=G)
    inp = synth.decode_inputs(wl, steps=6)
    assert inp["B"].shape == (6, 3, G, 2, 16)
    kw = dict(batch=3, H=4, P=8, N=16, R=2, dtype="bf16", steps=6)
    out = oracle.decode(inp, **kw)
    out2 = oracle.decode(dict(inp, B=_expand(inp["B"], 4), C=_expand(inp["C"], 4)), **kw)
    for a, b in zip(out, out2):
        assert np.array_equal(a, b)


def test_grouped_decode_continues_grouped_prefill():
    """Prefill then decode with grouped B/C gives the same outputs as one
    prefill over all tokens (the carry hands the group's last B over)."""
    H, P, N, R, L, T = 4, 8, 16, 1, 24, 5
    wl = synth.Workload("t", "prefill", 1, L + T, H, P, N, R, "bf16", chunk=16, ngroups=2)
    inp = synth.prefill_inputs(wl)
    kw = dict(batch=1, H=H, P=P, N=N, R=R, dtype="bf16", nthreads=1)
    y_all, _, _, _, _ = oracle.prefill(inp, L=L + T, **kw)
    head = {k: (v if k in ("A", "D") else v[:, :L]) for k, v in inp.items()}
    _, h, pB, px, _ = oracle.prefill(head, L=L, **kw)
    dec = {k: np.ascontiguousarray(np.swapaxes(v[:, L:], 0, 1)) for k, v in inp.items() if k not in ("A", "D")}
    dec.update(A=inp["A"], D=inp["D"], h0=h, prev_B=pB, prev_x=px)
    y_dec, _, _, _ = oracle.decode(dec, steps=T, **kw)
    assert np.allclose(y_dec[:, 0], y_all[0, L:], rtol=1e-9, atol=1e-9)
