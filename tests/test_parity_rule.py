"""CPU checks of the per-segment acceptance rule the GPU parity tests use.

The failure mode of TransformerEngine PR #671 (Verification) hides in later,
smaller segments while the whole tensor looks right, so every segment with
signal is judged on its own scale; only a segment whose exact gradient is zero
(fp64 round-off in the reference) is judged against the tensor's scale."""
import torch

from tests.parity import ZERO_SIGNAL_REL, call_scale, compare, per_segment_report


def _tensor(seed, rows):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(rows, 2, 8, generator=g, dtype=torch.float64)


def test_small_segment_with_signal_is_judged_on_its_own_scale():
    cu = [0, 40, 50]
    ref = _tensor(1, 50)
    ref[40:] *= 0.1            # a later segment with a tenth of the signal
    got = ref.clone()
    noise = _tensor(2, 10)
    got[40:] += 0.05 * float(ref[40:].abs().max()) * noise / float(noise.abs().max())
    # 5 % of the segment's own scale is only 0.5 % of the tensor's: the old
    # tensor-scale bound accepted it, the segment rule must not
    whole = compare(got, ref, 2e-2, 0.9999)
    assert whole["max_err"] <= 2e-2 * whole["max_ref"]
    rep = per_segment_report(got, ref, cu, "dq", 2e-2, 0.9999)
    assert [r["ok"] for r in rep] == [True, False]


def test_cosine_is_required_on_every_segment_with_signal():
    cu = [0, 30, 60]
    ref = _tensor(3, 60)
    ref[30:] *= 0.05
    got = ref.clone()
    got[30:] = ref[30:].flip(0)   # right magnitude everywhere, wrong values
    rep = per_segment_report(got, ref, cu, "dk", 2e-2, 0.9999)
    assert rep[0]["ok"] and not rep[1]["ok"] and rep[1]["cos"] < 0.9999


def test_zero_signal_segment_accepts_rounding_noise_at_tensor_scale():
    cu = [0, 20, 21]
    ref = _tensor(4, 21)
    ref[20:] = 1e-16 * ref[20:]        # exact zero up to fp64 round-off
    got = ref.clone()
    got[20:] = 1e-4 * float(ref.abs().max())   # fp32-level residue of a cancellation
    rep = per_segment_report(got, ref, cu, "dq", 2e-2, 0.9999)
    assert all(r["ok"] for r in rep)
    assert rep[1]["zero_signal"] and not rep[0]["zero_signal"]
    # above the round-off threshold the same segment is judged on its own scale
    ref[20:] = 10 * ZERO_SIGNAL_REL * float(ref.abs().max())
    rep = per_segment_report(got, ref, cu, "dq", 2e-2, 0.9999)
    assert not rep[1]["ok"]


def test_all_zero_reference_needs_exact_zeros_without_a_floor():
    z = torch.zeros(5, 2, 8, dtype=torch.float64)
    assert compare(z, z, 2e-2, 0.9999)["ok"]
    assert not compare(z + 1e-30, z, 2e-2, 0.9999)["ok"]


def test_fp32_rule_has_no_cosine_and_a_tight_bound():
    ref = _tensor(5, 10)
    assert compare(ref * (1 + 5e-5), ref, 1e-4, 0.0)["ok"]
    assert not compare(ref * (1 + 5e-4), ref, 1e-4, 0.0)["ok"]


def test_zero_gradient_tensor_is_judged_on_the_call_scale():
    """A single visible key per row: dQ and dK are exactly zero (dS = P (dP - D)
    cancels) while dV = sum of dO is not.  The kernel's fp32 residue of that
    cancellation is judged at the call's largest gradient; an error of 5 % of
    that scale still fails, and without a call scale the strict rule stays."""
    dv = _tensor(5, 20)
    dq = 1e-17 * _tensor(6, 20)               # exact zero up to fp64 round-off
    cf = call_scale([dq, dv])
    assert cf == float(dv.abs().max())
    residue = dq + 1e-7 * cf * _tensor(7, 20) / float(_tensor(7, 20).abs().max())
    rep = compare(residue, dq, 2e-2, 0.9999, cf)
    assert rep["ok"] and rep["zero_signal"]
    assert not compare(dq + 0.05 * cf, dq, 2e-2, 0.9999, cf)["ok"]
    assert not compare(residue, dq, 2e-2, 0.9999)["ok"]
    # a tensor with signal keeps its own scale even with a call scale given
    got = dv.clone()
    got[0, 0, 0] += 0.05 * float(dv.abs().max())
    assert not compare(got, dv, 2e-2, 0.9999, 10 * cf)["ok"]
    # segments of a zero-signal tensor take the call scale too
    rep = per_segment_report(residue, dq, [0, 10, 20], "dq", 2e-2, 0.9999, call_floor=cf)
    assert all(r["ok"] and r["zero_signal"] for r in rep)
