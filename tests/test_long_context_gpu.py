"""Long-context workload: B=1, T=32768, H=16, Dk=Dv=128, bf16 inputs, fp32 state.

The chunked forward and the recurrent kernel run the whole problem on the GPU;
the oracle checks all 16 heads over all 32768 tokens. Then the out-of-region
slice: one 64-token chunk whose keys are not normalised (beta |k|^2 ~ beta Dk
>> 2, the regime where the "gated-deltanet" card says the rule diverges),
started from the oracle's own final state, for all 16 heads.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_gdn_gb300 as gdn
import oracle
from gated_deltanet_gdn_gb300.synthetic import WORKLOADS, make_inputs, out_of_region_slice, to_f64

from helpers import TOL, head_slice, rel

pytestmark = pytest.mark.gpu
PAIRS = [(0, h) for h in range(16)]  # every head of the B1 H16 workload


@pytest.fixture(scope="module")
def long_run():
    w = WORKLOADS["long_context"]
    host = make_inputs(w)
    d = {k: (None if v is None else v.cuda()) for k, v in host.items()}
    out, hT, _ = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    ro, rh = gdn.gdn_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    torch.cuda.synchronize()
    args = [to_f64(head_slice(host[n], PAIRS, state=(n == "h0"))) for n in ("q", "k", "v", "g", "beta", "h0")]
    o_ref, h_ref = oracle.fwd(*args)
    return w, host, out.cpu(), hT.cpu(), ro.cpu(), rh.cpu(), o_ref, h_ref


def _report(label, out, hT, o_ref, h_ref):
    o = head_slice(out, PAIRS).double().numpy()
    h = head_slice(hT, PAIRS, state=True).double().numpy()
    per_o = [np.linalg.norm(o[0, :, i] - o_ref[0, :, i]) / np.linalg.norm(o_ref[0, :, i]) for i in range(len(PAIRS))]
    per_h = [np.linalg.norm(h[0, i] - h_ref[0, i]) / np.linalg.norm(h_ref[0, i]) for i in range(len(PAIRS))]
    whole_o, whole_h = rel(head_slice(out, PAIRS), o_ref), rel(head_slice(hT, PAIRS, state=True), h_ref)
    print(f"\n{label}: out {whole_o:.3e} (worst head {max(per_o):.3e}), "
          f"h_final {whole_h:.3e} (worst head {max(per_h):.3e})")
    return whole_o, whole_h, max(per_o), max(per_h)


def test_long_context_chunked_forward(long_run):
    """Every head, rel-L2 <= 2e-2 over the whole tensor and per head."""
    w, host, out, hT, ro, rh, o_ref, h_ref = long_run
    whole_o, whole_h, head_o, head_h = _report("long context chunked bf16", out, hT, o_ref, h_ref)
    assert max(whole_o, head_o) <= TOL["bf16"] and max(whole_h, head_h) <= TOL["bf16"]
    assert bool(torch.isfinite(out.float()).all()) and bool(torch.isfinite(hT).all())


def test_long_context_recurrent(long_run):
    """Every head: out within the bf16 tolerance (bf16 output), the fp32 final state
    within 1e-4 (exact recurrence in fp32), per head."""
    w, host, out, hT, ro, rh, o_ref, h_ref = long_run
    whole_o, whole_h, head_o, head_h = _report("long context recurrent", ro, rh, o_ref, h_ref)
    assert max(whole_o, head_o) <= TOL["bf16"]
    assert max(whole_h, head_h) <= 1e-4


def _perturbed_runs(args, rel, trials=8, seed=0):
    """The exact rule on this slice with q, k, v and the incoming state given
    i.i.d. relative perturbations of size `rel`, over `trials` seeded draws."""
    rng = np.random.default_rng(seed)
    runs = []
    for _ in range(trials):
        b = list(args)
        for i in (0, 1, 2, 5):
            b[i] = args[i] * (1 + rng.uniform(-rel, rel, args[i].shape))
        runs.append(oracle.fwd(*b)[0])
    return runs


def _row_envelope(args, ref, rel):
    """Per output row, the largest relative deviation of a perturbed run: how far
    the exact rule itself moves when its inputs carry errors of size `rel`."""
    norms = np.linalg.norm(ref, axis=-1)
    env = np.zeros_like(norms)
    with np.errstate(all="ignore"):
        for p in _perturbed_runs(args, rel):
            dev = np.linalg.norm(p - ref, axis=-1) / np.maximum(norms, 1e-30)
            env = np.maximum(env, np.where(np.isfinite(dev), dev, 0.0))
    return env


def _aggregate_envelope(args, ref, rel):
    """Largest per-row |log10 norm ratio| and largest aggregate relative error of
    a perturbed run over the rows where the exact result is finite."""
    norms = np.linalg.norm(ref, axis=-1)
    worst_ratio = worst_agg = 0.0
    with np.errstate(all="ignore"):
        for p in _perturbed_runs(args, rel):
            ok = np.isfinite(ref).all(-1) & (norms < 1e30) & np.isfinite(p).all(-1)
            worst_ratio = max(worst_ratio, np.abs(np.log10(np.linalg.norm(p, axis=-1)[ok] / norms[ok])).max())
            worst_agg = max(worst_agg, np.linalg.norm((p - ref)[ok]) / np.linalg.norm(ref[ok]))
    return worst_ratio, worst_agg


def _divergence_check(o_gpu, o_ref, tol, env):
    """Per-row rule: within max(tol, the row's perturbation envelope) while the
    oracle row norm stays below 1e30; non-finite once the oracle row leaves the
    fp32 range. Returns the rows checked, the rows required non-finite, the largest
    bound used and how many rows the envelope widened beyond tol."""
    o = o_gpu.double().numpy()
    checked = nonfinite = widened = 0
    largest = tol
    for t in range(o.shape[1]):
        for h in range(o.shape[2]):
            ref = o_ref[0, t, h]
            nrm = np.linalg.norm(ref)
            if nrm < 1e30:
                err = np.linalg.norm(o[0, t, h] - ref) / max(nrm, 1e-30)
                bound = max(tol, env[0, t, h])
                assert err <= bound, (t, h, err, env[0, t, h])
                checked += 1
                widened += int(bound > tol)
                largest = max(largest, bound)
            elif not np.isfinite(nrm) or nrm > 3.4e38:
                assert not np.all(np.isfinite(o[0, t, h])), (t, h)
                nonfinite += 1
    return checked, nonfinite, largest, widened


def _early_rows(o_gpu, o_ref, growth=1e3):
    """Per-row rel-L2 of every head's rows before the oracle's output norm first grows
    past `growth` times its first row's, and the rel-L2 over all of them together."""
    o = o_gpu.double().numpy()
    errs, num, den = [], 0.0, 0.0
    for h in range(o.shape[2]):
        n0 = np.linalg.norm(o_ref[0, 0, h])
        for t in range(o.shape[1]):
            ref = o_ref[0, t, h]
            nrm = np.linalg.norm(ref)
            if not nrm < growth * n0:
                break
            diff = np.linalg.norm(o[0, t, h] - ref)
            errs.append(diff / nrm)
            num, den = num + diff ** 2, den + nrm ** 2
    return np.array(errs), float(np.sqrt(num / den))


def test_out_of_region_slice_diverges_like_the_oracle(long_run):
    """The pages give no accuracy for any form of the rule in this regime, and on
    this slice the rule is badly conditioned: relative input perturbations of one
    fp32 unit roundoff already move single rows by ~5e-4, bf16-sized ones by ~10x
    in norm. So each tolerance is the output's tolerance or the spread of eight
    seeded perturbed oracle runs, whichever is larger, with the perturbation set
    by the arithmetic: Dk * 2^-24 (the dot-product rounding bound in fp32) for the
    recurrent kernel and the fp32 chunked path, checked row by row; 2^-9 (bf16
    operands) for the bf16 chunked path, checked by per-row norm ratio and in
    aggregate, after it has reproduced the divergence (growth by > 1e6). The bf16
    chunked path is NOT held to a per-row bound: it rounds the state and the WY
    factors to bf16 as tensor-core operands, and single rows that cancel inside
    amplify that rounding (measured before any growth, at row 0 of some heads, up to
    ~3e-2; beyond 2e-2 on about a quarter of the rows before a thousandfold growth),
    so no per-row bound at the bf16 tolerance holds there; its per-row errors on
    those early rows are printed as a measurement. The largest bound used and the
    number of rows whose bound the envelope widened are printed for the checked
    paths."""
    w, host, out, hT, ro, rh, o_ref, h_ref = long_run
    h0 = torch.from_numpy(h_ref).to(torch.float32)  # the oracle's state after the region
    for dtype in ("bf16", "f32"):
        sl = out_of_region_slice(w.with_(H=len(PAIRS), dtype=dtype), h0)
        args = [to_f64(sl[n]) for n in ("q", "k", "v", "g", "beta", "h0")]
        so_ref, _ = oracle.fwd(*args)
        norms = np.linalg.norm(so_ref, axis=-1)
        assert norms.max() > 1e6 * norms[:, :2].max()  # the slice does diverge
        d = {k: (None if v is None else v.cuda()) for k, v in sl.items()}
        r_out, _ = gdn.gdn_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
        c_out, _, _ = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
        torch.cuda.synchronize()
        env = _row_envelope(args, so_ref, w.Dk * 2.0 ** -24)
        checked, nonfin, largest, widened = _divergence_check(r_out.cpu(), so_ref, TOL[dtype], env)
        print(f"\nout-of-region {dtype} recurrent: {checked} rows checked ({widened} with the bound widened "
              f"beyond {TOL[dtype]:g}, largest bound {largest:.3e}), {nonfin} rows non-finite as required")
        assert checked > 0
        if dtype == "f32":
            checked, nonfin, largest, widened = _divergence_check(c_out.cpu(), so_ref, TOL["f32"], env)
            print(f"out-of-region f32 chunked: {checked} rows checked ({widened} widened beyond 1e-4, "
                  f"largest bound {largest:.3e}), {nonfin} rows non-finite as required")
        else:
            finite = np.isfinite(so_ref).all(axis=-1) & (norms < 1e30)
            co = c_out.double().cpu().numpy()
            cn = np.linalg.norm(co, axis=-1)
            assert cn[finite].max() > 1e6 * cn[:, :2].max()  # the chunked path diverges too
            errs, early = _early_rows(c_out.cpu(), so_ref)
            env_ratio, env_agg = _aggregate_envelope(args, so_ref, 2.0 ** -9)
            ratio = np.abs(np.log10(cn[finite] / norms[finite])).max()
            err = np.linalg.norm((co - so_ref)[finite]) / np.linalg.norm(so_ref[finite])
            # measured, not asserted: no per-row bound at the bf16 tolerance holds for the
            # bf16 chunked path in this regime (rows before growth included)
            print(f"out-of-region bf16 chunked: {len(errs)} early rows (before 1e3 growth): rel-L2 over them "
                  f"{early:.3e}, median row {np.median(errs):.3e}, worst row {errs.max():.3e}, "
                  f"{int((errs > TOL['bf16']).sum())} rows above 2e-2; norm ratio {ratio:.3f} decades "
                  f"(envelope {env_ratio:.3f}); aggregate {err:.3e} (envelope {env_agg:.3e})")
            assert len(errs) > 0
            assert ratio <= env_ratio, (ratio, env_ratio)
            assert err <= env_agg, (err, env_agg)
            checked = int(finite.sum())
        assert checked > 0
