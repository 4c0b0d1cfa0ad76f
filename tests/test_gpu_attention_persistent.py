"""Joint attention [klein, section 4.3] under the persistent schedule (dit_attention_workspace_bytes).

When the (query-tile pair, head) units leave the last wave over the SMs part-empty, one CTA per SM
takes an equal share of all the units' key tiles and a unit cut between two CTAs is finished by the
one that holds its first key tiles, from the unnormalised partial the other leaves in the scratch.
Checked here on shapes with cut units, in the three softmax paths (fixed maximum with unit weights,
fixed maximum chosen on the device from near-one weights, running maximum):

* against the float64 oracle (all rows, or sampled rows at the full 1024sq size);
* against the same call without scratch (one CTA per unit): bit for bit on the rows of units that
  stay whole (the same arithmetic in the same order); on the cut units within one bf16 step under a
  fixed maximum (the same weights, two fp32 partial sums added once), within the oracle's bound
  under a running maximum (each part rounds its weights to bf16 against its own maximum);
* repeated launches (more than the ready words' slot blocks) give the same bits: the result does
  not depend on timing.
"""

import numpy as np
import pytest
import torch

import dit_inputs as DI
import diffusion_transformer_gb300 as D
import oracle as O
from tests.gpu_util import bf16_f64, dev, dev_bf16, max_abs

pytestmark = pytest.mark.gpu


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _cut_units(R, nh):
    """Units (head * pairs + pair) that the schedule divides between two CTAs, or None if the shape
    runs one CTA per unit on this GPU."""
    nkv = (R + 127) // 128
    npairs = (nkv + 1) // 2
    units = nh * npairs
    sms = _sms()
    if units <= sms or units % sms == 0:
        return None
    total = units * nkv
    work = -(-total // sms)
    ctas = -(-total // work)
    cut = set()
    for c in range(1, ctas):
        b = c * work
        if b % nkv:
            cut.add(b // nkv)
    return sorted(cut), npairs


def _qknormed(g, nh, R, d, w):
    x = g.standard_normal((nh, R, d))
    x = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + 1e-6)
    if w is not None:
        x = x * w
    return DI.bf16_bits_from_f32(x.astype(np.float32))


def _case(R, nh, d, mode, seed):
    g = np.random.default_rng(seed)
    w = None
    if mode == "auto":
        w = (1 + 0.02 * g.standard_normal(d)).astype(np.float32)
    q, k = _qknormed(g, nh, R, d, w), _qknormed(g, nh, R, d, w)
    v = DI.bf16_bits_from_f32(g.standard_normal((nh, R, d), dtype=np.float32))
    vt = np.zeros((nh, d, D.dit_vt_stride(R)), np.uint16)
    vt[:, :, :R] = v.transpose(0, 2, 1)
    return q, k, v, vt, w


def _run(dims, R, q, k, vt, w, mode, ws):
    o = torch.empty(R, dims.heads * dims.head_dim, dtype=torch.bfloat16, device="cuda")
    if mode == "running":
        D.dit_attention(dims, R, q, k, vt, o, ws=ws)
    else:
        wd = None if w is None else dev(w)
        D.dit_attention_qknorm(dims, R, q, k, vt, wd, wd, o, ws=ws)
    D.dit_check()
    return o


@pytest.mark.parametrize("R,nh,d", [(2000, 24, 128), (1000, 48, 64), (4224, 24, 128)])
@pytest.mark.parametrize("mode", ["fixed", "auto", "running"])
def test_persistent_attention(R, nh, d, mode):
    plan = _cut_units(R, nh)
    if plan is None:
        pytest.skip("this GPU's SM count fills the last wave: one CTA per unit")
    cut, npairs = plan
    assert cut, "no unit is cut: the partial path would go untested"
    dims = D.DitDims(nh * d, nh, d, 256)
    need = D.dit_attention_workspace_bytes(dims, R)
    assert need > 0
    q, k, v, vt, w = _case(R, nh, d, mode, R + nh + len(mode))
    qd, kd, vtd = dev_bf16(q), dev_bf16(k), dev_bf16(vt)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    o_p = _run(dims, R, qd, kd, vtd, w, mode, ws)
    o_u = _run(dims, R, qd, kd, vtd, w, mode, None)

    # against the oracle: every row, or 256 sampled rows (always including some of the cut units)
    f = lambda a: O.bf16_to_f64(a).transpose(1, 0, 2)
    g = np.random.default_rng(7)
    if R * nh <= 48000:
        rows = np.arange(R)
    else:
        rows = np.unique(np.concatenate([g.choice(R, 192, replace=False),
                                         [min(R - 1, (u % npairs) * 256 + 5) for u in cut[:16]]]))
    qf, kf, vf = f(q), f(k), f(v)
    ref = O.attention(qf, kf, vf, rows=rows)
    vmax = np.abs(vf).max()
    for got in (bf16_f64(o_p)[rows], bf16_f64(o_u)[rows]):
        assert np.all(np.abs(got - ref) <= 2 ** -8 * vmax + 2 ** -8 * np.abs(ref)), max_abs(got, ref)

    # against the unscheduled launch: whole units bit for bit, cut units within one bf16 step
    a, b = bf16_f64(o_p), bf16_f64(o_u)
    in_cut = np.zeros((R, nh), bool)
    for u in cut:
        head, qp = divmod(u, npairs)
        in_cut[qp * 256:min(R, qp * 256 + 256), head] = True
    mask = np.repeat(in_cut, d, axis=1)
    assert np.array_equal(a[~mask], b[~mask])
    diff = np.abs(a[mask] - b[mask])
    if mode == "running":
        # each part of a cut unit keeps its own running maximum, so its weights exp2(s - m) are
        # rounded to bf16 at another scale than in the whole row: the bound of the oracle check
        assert np.all(diff <= 2 ** -8 * vmax + 2 ** -8 * np.abs(b[mask])), float(diff.max())
    else:
        # the same weights; two fp32 partial sums added once: one bf16 step of the value (8
        # significant bits: at most 2^-7 of it)
        assert np.all(diff <= 2 ** -7 * np.abs(b[mask]) + 2 ** -20 * vmax), float(diff.max())
    print(f"R={R} heads={nh} d={d} {mode}: {len(cut)} cut units, "
          f"{np.count_nonzero(diff)} of {diff.size} cut-unit values differ from the unscheduled launch")

    # launches past the 64 slot blocks of ready words: the same bits every time
    if R == 2000 and mode == "fixed":
        for _ in range(70):
            o_again = _run(dims, R, qd, kd, vtd, w, mode, ws)
            assert torch.equal(o_again, o_p)


def test_persistent_attention_scratch_too_small_runs_one_cta_per_unit():
    R, nh, d = 2000, 24, 128
    if _cut_units(R, nh) is None:
        pytest.skip("this GPU's SM count fills the last wave")
    dims = D.DitDims(nh * d, nh, d, 256)
    q, k, v, vt, w = _case(R, nh, d, "fixed", 3)
    qd, kd, vtd = dev_bf16(q), dev_bf16(k), dev_bf16(vt)
    small = torch.zeros(D.dit_attention_workspace_bytes(dims, R) - 16, dtype=torch.uint8, device="cuda")
    assert torch.equal(_run(dims, R, qd, kd, vtd, w, "fixed", small), _run(dims, R, qd, kd, vtd, w, "fixed", None))


def test_persistent_attention_replayed_in_a_cuda_graph():
    # a captured launch keeps its epoch across replays: every replay must still wait for the partials
    # of its own run (the finisher clears the ready word it consumed), so each replay on fresh inputs
    # equals a direct call on them bit for bit
    R, nh, d = 2000, 24, 128
    if _cut_units(R, nh) is None:
        pytest.skip("this GPU's SM count fills the last wave")
    dims = D.DitDims(nh * d, nh, d, 256)
    q0, k0, v0, vt0, w = _case(R, nh, d, "fixed", 11)
    qd, kd, vtd = dev_bf16(q0), dev_bf16(k0), dev_bf16(vt0)
    ws = torch.zeros(D.dit_attention_workspace_bytes(dims, R), dtype=torch.uint8, device="cuda")
    o = torch.empty(R, nh * d, dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        D.dit_attention_qknorm(dims, R, qd, kd, vtd, None, None, o, ws=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        D.dit_attention_qknorm(dims, R, qd, kd, vtd, None, None, o, ws=ws)
    for seed in (12, 13, 14, 15):
        q, k, v, vt, _ = _case(R, nh, d, "fixed", seed)
        qd.copy_(dev_bf16(q))
        kd.copy_(dev_bf16(k))
        vtd.copy_(dev_bf16(vt))
        graph.replay()
        torch.cuda.synchronize()
        direct = _run(dims, R, dev_bf16(q), dev_bf16(k), dev_bf16(vt), None, "fixed",
                      torch.zeros_like(ws))
        assert torch.equal(o, direct), seed
    D.dit_check()
