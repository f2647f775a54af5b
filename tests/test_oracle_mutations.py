"""Planted mistakes in a copy of the oracle must each fail at least one pin.

The copy is made from the oracle's source text with one plausible error
inserted (a dropped term, a wrong sign or index, a wrong operand); it runs on
the CPU only.  The pins re-run here are the independent ones from
test_oracle_pins: brute force, torch SDPA on single documents, and finite
differences.
"""
import os
import types

import numpy as np
import pytest

import test_oracle_dropout as dpins
import test_oracle_pins as pins
import test_oracle_row_slices as spins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "blockdiag.py")

MUTATIONS = {
    "causal_off_by_one": ("keys[None, :] <= np.arange(r0, r1)[:, None]",
                          "keys[None, :] <= np.arange(r0, r1)[:, None] + 1"),
    "cross_document": ("if ids[p] != ids[p - 1]]", "if ids[p] != ids[p - 1] and ids[p] == 0]"),
    "gqa_modulo": ("g = h // G", "g = h % Hkv"),
    "pad_not_masked": ("if sid == PAD_DOC_ID:\n                continue",
                       "if False:\n                continue"),
    "lse_without_log": ("row_lse = m + np.log(np.exp(s - m).sum(axis=1, keepdims=True))",
                        "row_lse = m + np.exp(s - m).sum(axis=1, keepdims=True) - 1.0"),
    "dq_missing_scale": ("dq[b, h, i0:i1] = scale * (ds @ kk)", "dq[b, h, i0:i1] = ds @ kk"),
    "ds_sign": ("ds = p * (dp - delta[b, h, i0:i1, None])",
                "ds = p * (dp + delta[b, h, i0:i1, None])"),
    "dv_into_dk": ("dv[b, g, start:r1] += pd.T @ dout[b, h, i0:i1]",
                   "dk[b, g, start:r1] += pd.T @ dout[b, h, i0:i1]"),
    "dk_uses_k": ("dk[b, g, start:r1] += scale * (ds.T @ q[b, h, i0:i1])",
                  "dk[b, g, start:r1] += scale * (ds.T @ q[b, h, i0:i1][:, ::-1])"),
    "dropout_unscaled": ("dropout_p) * keep_scale(dropout_p)\n                    out[b, h",
                         "dropout_p)\n                    out[b, h"),
    "dropout_dv_undropped": ("dv[b, g, start:r1] += pd.T @ dout[b, h, i0:i1]",
                             "dv[b, g, start:r1] += p.T @ dout[b, h, i0:i1]"),
    "dropout_ds_unmasked": ("                        pd, dp = p * mr, dp * mr",
                            "                        pd = p * mr"),
    "dropout_mask_local_rows": (
        "p = p * keep_mask(_mask_plane(mask_planes, b, h, Hq),\n"
        "                                          np.arange(r0, r1) + mask_pos0",
        "p = p * keep_mask(_mask_plane(mask_planes, b, h, Hq),\n"
        "                                          np.arange(r0, r1) - seq_start + mask_pos0"),
    "interval_offset": ("q[b, h, r0 - seq_start:r1 - seq_start] @ k[b, g, start:r1].T",
                        "q[b, h, r0:r1] @ k[b, g, start:r1].T"),
    # mistakes that only show once a segment is cut into several row slices
    "slices_overlap": ("yield t, min(t1, t + step)", "yield t, min(t1, t + step + 1)"),
    "slice_rows_from_first_slice": (
        "q[b, h, r0 - seq_start:r1 - seq_start] @ k[b, g, start:r1].T",
        "q[b, h, t0 - seq_start:t0 - seq_start + r1 - r0] @ k[b, g, start:r1].T"),
    "slice_dropout_rows_from_first_slice": (
        "p = p * keep_mask(_mask_plane(mask_planes, b, h, Hq),\n"
        "                                          np.arange(r0, r1) + mask_pos0",
        "p = p * keep_mask(_mask_plane(mask_planes, b, h, Hq),\n"
        "                                          np.arange(t0, t0 + r1 - r0) + mask_pos0"),
}


def _mutant(name):
    src = open(SRC).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    src = src.replace(old, new).replace("from .dropout import", "from oracle.dropout import")
    exec(compile(src, SRC, "exec"), mod.__dict__)
    return mod


def _pins(orc, monkeypatch):
    monkeypatch.setattr(pins, "orc", orc)
    monkeypatch.setattr(dpins, "orc", orc)
    checks = [
        lambda: pins.test_golden_tiny_segments(),
        lambda: pins.test_golden_padded_small(),
        lambda: pins.test_forward_matches_brute_force(
            ([[4, 4, 4, 4, 4, 7, 7, 7, 0, 0, 9, 9]], 3, 6, 4, 2, 2)),
        lambda: pins.test_forward_matches_brute_force(
            ([[1, 1, 2, 2, 1, 1, 0, 0]], 0, 8, 2, 2, 4)),
        lambda: pins.test_single_document_is_torch_causal_sdpa(8),
        lambda: pins.test_packed_equals_documents_run_separately(),
        lambda: pins.test_backward_matches_finite_differences(),
        lambda: dpins.test_dropout_forward_matches_dense_statement(dpins.CASES[1]),
        lambda: dpins.test_dropout_backward_matches_finite_differences(),
        lambda: dpins.test_dropout_intervals_concatenate_to_full_rows(),
    ] + [
        (lambda n=n, b=b: spins.check_sliced_oracle(orc, n, b))
        for n in sorted(spins.CASES) for b in (5, 256)
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except (AssertionError, IndexError, ValueError, FloatingPointError):
            failed += 1
    return failed


def test_unmutated_oracle_passes_all(monkeypatch):
    src = open(SRC).read().replace("from .dropout import", "from oracle.dropout import")
    mod = types.ModuleType("oracle_copy")
    exec(compile(src, SRC, "exec"), mod.__dict__)
    assert _pins(mod, monkeypatch) == 0


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    with np.errstate(all="ignore"):
        assert _pins(_mutant(name), monkeypatch) >= 1
