"""Helpers shared by the GPU parity tests: moving bf16 bit patterns to the
device and comparing GPU outputs with the oracle's."""
import numpy as np
import torch


def to_device(bits, device="cuda"):
    """uint16 bf16 bit patterns (numpy) -> torch.bfloat16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def host(t):
    return t.cpu().numpy()


def assert_equal_bytes(got, want, what):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        first = [tuple(int(i) for i in b) for b in bad[:5]]
        vals = [(int(got[b]), int(want[b])) for b in first]
        raise AssertionError(f"{what}: {len(bad)} of {got.size} differ; first {first} "
                             f"(got, want) = {vals}")


def e4m3_ordinal(codes):
    """Signed position of an E4M3 code on the number line (+-0 -> 0)."""
    c = np.asarray(codes).astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def check_activation_blocks(q, s, q_ref, s_ref, block_axis, what, code_frac=1e-4, scale_frac=1e-4):
    """Tolerance check for the fused-activation paths (y computed in fp32 on
    the GPU, in double rounded to fp32 by the oracle): scale codes may differ
    in at most scale_frac of the blocks, by one; in blocks whose scales agree,
    at most code_frac of the elements may differ, each by one E4M3 step.
    block_axis: axis of q along which consecutive 32 elements share a scale
    (1 for [rows][cols] layouts, which both rowwise and colwise outputs use)."""
    q, s, q_ref, s_ref = map(np.asarray, (q, s, q_ref, s_ref))
    assert q.shape == q_ref.shape and s.shape == s_ref.shape
    sdiff = s.astype(np.int32) - s_ref.astype(np.int32)
    assert np.all(np.abs(sdiff) <= 1), f"{what}: a scale differs by more than one"
    n_sbad = int(np.count_nonzero(sdiff))
    assert n_sbad <= max(1, scale_frac * s.size), f"{what}: {n_sbad} of {s.size} scales differ"
    same_scale = np.repeat(sdiff == 0, 32, axis=block_axis)
    d = np.abs(e4m3_ordinal(q) - e4m3_ordinal(q_ref))
    d = np.where(same_scale, d, 0)
    assert d.max(initial=0) <= 1, f"{what}: a code differs by more than one step"
    n_bad = int(np.count_nonzero(d))
    assert n_bad <= max(1, code_frac * q.size), f"{what}: {n_bad} of {q.size} codes differ"
    return n_bad, n_sbad


def count_activation_mismatches(q, s, q_ref, s_ref, chunk_rows=1024):
    """Whole-tensor counts for the fused-activation tolerance, taken in row
    chunks (blocks run along axis 1 in every layout, so a row chunk holds
    whole blocks): the largest scale difference and the number of differing
    scales; over blocks whose scales agree, the largest code difference in
    E4M3 steps and the number of differing codes."""
    q, s, q_ref, s_ref = map(np.asarray, (q, s, q_ref, s_ref))
    assert q.shape == q_ref.shape and s.shape == s_ref.shape
    res = {"codes": int(q.size), "scales": int(s.size), "max_scale_diff": 0, "scales_differ": 0,
           "max_code_steps": 0, "codes_differ": 0}
    for r0 in range(0, q.shape[0], chunk_rows):
        r1 = min(q.shape[0], r0 + chunk_rows)
        sd = s[r0:r1].astype(np.int32) - s_ref[r0:r1].astype(np.int32)
        res["max_scale_diff"] = max(res["max_scale_diff"], int(np.abs(sd).max(initial=0)))
        res["scales_differ"] += int(np.count_nonzero(sd))
        same = np.repeat(sd == 0, 32, axis=1)
        d = np.abs(e4m3_ordinal(q[r0:r1]) - e4m3_ordinal(q_ref[r0:r1]))
        d = np.where(same, d, 0)
        res["max_code_steps"] = max(res["max_code_steps"], int(d.max(initial=0)))
        res["codes_differ"] += int(np.count_nonzero(d))
    res["code_frac"] = res["codes_differ"] / max(1, res["codes"])
    res["scale_frac"] = res["scales_differ"] / max(1, res["scales"])
    return res


def assert_activation_budget(res, what, frac=1e-4):
    """The fused-activation contract over a whole tensor: scales within one
    code and codes within one E4M3 step, each differing in at most `frac`
    of the tensor."""
    assert res["max_scale_diff"] <= 1, f"{what}: a scale differs by {res['max_scale_diff']}"
    assert res["max_code_steps"] <= 1, f"{what}: a code differs by {res['max_code_steps']} steps"
    assert res["scale_frac"] <= frac, f"{what}: {res['scales_differ']} of {res['scales']} scales differ"
    assert res["code_frac"] <= frac, f"{what}: {res['codes_differ']} of {res['codes']} codes differ"


def record(what, **numbers):
    """Print a measured parity figure; with MXQ_PARITY_LOG set, also append
    it as one JSON line to that file."""
    import json
    import os

    line = json.dumps({"case": what, **numbers})
    print(line)
    path = os.environ.get("MXQ_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")
