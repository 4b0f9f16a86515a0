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
