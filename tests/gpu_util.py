"""Helpers of the GPU parity tests: compare what the CUDA path returned (through
the C ABI binding) with the fp64 oracle.  The upload helpers live in
synth.device (the benchmark and smoke() use them too) and are re-exported
here for the tests."""
from __future__ import annotations

import json

import numpy as np

import compare
import synth
from synth.device import GqaDev, MlaDev, bits, dev  # noqa: F401  (re-exported for the tests)


def gqa_oracle(w: synth.GQAWorkload, rows=None, window=None):
    import oracle
    return oracle.gqa(w.q, w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale,
                      w.window if window is None else window, rows=rows)


def check_gqa(w, out_bits, lse, rows=None, window=None, tol_abs=compare.MAX_ABS, tol_rel=compare.MAX_REL):
    """Compare GPU output (all rows, or the sampled (b, h) rows) with the oracle; return stats."""
    B, Hq, D = w.q.shape
    ro, rl = gqa_oracle(w, rows, window)
    if rows is None:
        got_o = out_bits.reshape(-1, D)
        got_l = lse.reshape(-1)
    else:
        idx = np.asarray(rows)
        got_o = out_bits[idx[:, 0], idx[:, 1]]
        got_l = lse[idx[:, 0], idx[:, 1]]
    st = compare.compare(got_o, ro)
    dl = compare.lse_max_abs(got_l, rl)
    assert st.max_abs <= tol_abs and st.max_rel <= tol_rel, f"{w.name}: {st}"
    assert dl <= compare.LSE_ABS, f"{w.name}: lse max abs err {dl:.3e}"
    return st, dl


def check_mla(w, out_bits, lse, rows=None):
    import oracle
    B, H, _ = w.q.shape
    ro, rl = oracle.mla(w.q, w.cache, w.w_uk, w.w_uv, w.layout.block_table, w.layout.context_lens, w.scale,
                        rows=rows)
    if rows is None:
        got_o = out_bits.reshape(-1, 128)
        got_l = lse.reshape(-1)
    else:
        idx = np.asarray(rows)
        got_o = out_bits[idx[:, 0], idx[:, 1]]
        got_l = lse[idx[:, 0], idx[:, 1]]
    st = compare.compare(got_o, ro)
    dl = compare.lse_max_abs(got_l, rl)
    assert st.max_abs <= compare.MAX_ABS and st.max_rel <= compare.MAX_REL, f"{w.name}: {st}"
    assert dl <= compare.LSE_ABS, f"{w.name}: lse max abs err {dl:.3e}"
    return st, dl


def report(name: str, shape, st: compare.Stats, lse_err: float) -> dict:
    """One line of the whole-tensor numerics table (the statistics of the kernel-numerics table
    of vllm.cpp PR #425, EVIDENCE section), printed with a NUMERICS prefix so a run with -s
    can collect the table; the worst element's index is unravelled over the output shape."""
    worst = tuple(int(x) for x in np.unravel_index(st.worst_index, shape)) if st.worst_index >= 0 else None
    rec = {"workload": name, "outputs": int(np.prod(shape[:-1])), "elements": st.n,
           "max_abs": float(f"{st.max_abs:.4g}"), "max_rel": float(f"{st.max_rel:.4g}"),
           "max_rel_elem": float(f"{st.max_rel_elem:.4g}"), "bitwise_pct": round(st.bitwise_pct, 3),
           "worst_index": worst, "lse_max_abs": float(f"{lse_err:.4g}")}
    print("NUMERICS " + json.dumps(rec), flush=True)
    return rec


def sample_rows(B, H, n, seed):
    u = synth.uniform01(seed, np.arange(2 * n, dtype=np.uint64))
    b = np.minimum((u[:n] * B).astype(np.int64), B - 1)
    h = np.minimum((u[n:] * H).astype(np.int64), H - 1)
    return [(int(x), int(y)) for x, y in zip(b, h)]
