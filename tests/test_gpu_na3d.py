"""GPU checks of rope3d_na3d (3D neighbourhood attention with the RoPE fused
into its prologue) and rope3d_na3d_rotate_once (K rotated once beforehand, Q
in the prologue) against the float64 oracle, and of the fusion itself: both
fused forms must give the same bits as the attention kernel fed with Q and K
rotated by rope3d_apply_pair.

Tolerance (derived from the arithmetic): the rotated operands are exact
bf16; scores accumulate in fp32; the probabilities are rounded to bf16
(relative 2^-9) before the tensor-core P.V product while the normaliser
uses the unrounded ones, and the output is rounded to bf16 (2^-9 of |O|):
|O - O_ref| <= 2^-7 * sum_k p_k |v_k| + 2^-8 |O_ref| + 1e-6, twice the
first-order bound."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU hosts
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import rope_rope3d_apply_gb300 as r  # noqa: E402

DEV = torch.device("cuda:0")

# The attention kernels: 1 = tensor-core (tcgen05; the default where its
# geometry allows), 2 = warp-level MMA. Each is held to the same bound.
KERNELS = [1, 2]


@pytest.fixture(autouse=True)
def _kernel_choice_and_no_timeouts():
    r.rope3d_testing_na3d_wait_timeouts(reset=True)
    yield
    r.rope3d_testing_na3d_kernel(0)
    r.rope3d_testing_na3d_per_cta(False)
    assert r.rope3d_testing_na3d_wait_timeouts(reset=True) == 0


def bf16(a):
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)


def to_f64(t):
    return (t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32).astype(np.float64)


CASES = [
    # (B, T, H, W, heads), split, kernel
    ((1, 3, 12, 12, 2), (32, 48, 48), (3, 5, 5)),
    ((2, 2, 9, 17, 1), (32, 48, 48), (1, 3, 7)),      # partial query blocks at both edges
    ((1, 5, 8, 8, 2), (48, 40, 40), (5, 7, 7)),        # windows covering the grid
    ((1, 4, 16, 24, 1), (32, 48, 48), (3, 7, 7)),
    ((1, 2, 6, 80, 1), (32, 48, 48), (1, 3, 67)),      # a region row of 74 keys: split in columns
    ((1, 2, 12, 40, 1), (32, 48, 48), (1, 9, 33)),     # region rows of 40 keys: three 16-key steps
    ((2, 4, 13, 11, 3), (16, 56, 56), (3, 5, 7)),      # two batches, three heads, odd grid, split
    ((2, 3, 9, 10, 2), (32, 48, 48), (3, 5, 5)),       # two batches, odd T: the last frame pair of
                                                        # batch 0 must not reach batch 1's first frame
    ((1, 1, 8, 8, 608), (32, 48, 48), (1, 3, 3)),      # 608 one-chunk blocks: four per CTA in turn
    ((1, 3, 8, 16, 96), (32, 48, 48), (3, 5, 5)),      # 384 blocks of one and two frames, several per CTA
    ((1, 2, 40, 24, 80), (32, 48, 48), (1, 7, 7)),     # 1,200 blocks: each CTA meets more window
                                                        # geometries than it keeps mask sets for
]


def attend(path, q, k, v, tabs, kernel):
    """The attention with the RoPE applied: rope3d_na3d (K rotated once into
    the library's scratch), the same with every K tile rotated per CTA, or
    rope3d_na3d_rotate_once (K rotated into the caller's buffer)."""
    if path in ("qk", "per_cta"):
        r.rope3d_testing_na3d_per_cta(path == "per_cta")
        return r.rope3d_na3d(q, k, v, tabs, kernel)
    return r.rope3d_na3d_rotate_once(q, k, v, tabs, kernel)[0]


PATHS = ["qk", "per_cta", "once"]


@pytest.mark.parametrize("which", KERNELS)
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[2]}" for c in CASES])
def test_na3d_matches_oracle(case, path, which):
    r.rope3d_testing_na3d_kernel(which)
    (B, T, H, W, heads), split, kernel = case
    shape6 = (B, T, H, W, heads, 128)
    n = int(np.prod(shape6))
    q_np = synthetic.normal(n, 1.0, 300, 0, "bf16")
    k_np = synthetic.normal(n, 1.0, 300, 1, "bf16")
    v_np = synthetic.normal(n, 1.0, 300, 2, "bf16")
    shp = (B, T * H * W, heads, 128)
    q, k, v = (bf16(a).reshape(shp).to(DEV) for a in (q_np, k_np, v_np))
    tabs = r.rope3d_build_tables(T, H, W, split)
    out = attend(path, q, k, v, tabs, kernel)
    torch.cuda.synchronize()
    assert r.rope3d_testing_na3d_last_kernel() == which
    got = to_f64(out).reshape(shape6)
    otabs = oracle.tables(T, H, W, split)
    ref = oracle.rope_na3d(q_np, k_np, v_np, shape6, split, otabs, kernel)
    qr = oracle.rope3d(q_np, shape6, split, otabs)
    kr = oracle.rope3d(k_np, shape6, split, otabs)
    vf = (v_np.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    to64 = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)  # noqa: E731
    absv = oracle.na3d(to64(qr), to64(kr), np.abs(vf), shape6, kernel)
    bound = 2.0 ** -7 * absv + 2.0 ** -8 * np.abs(ref) + 1e-6
    err = np.abs(got - ref)
    assert np.all(err <= bound), (err.max(), (err / bound).max())
    tabs.close()


@pytest.mark.parametrize("per_cta", [False, True])
@pytest.mark.parametrize("which", KERNELS)
def test_fused_equals_unfused_bitwise(which, per_cta):
    """The fused forms rotate exactly as rope3d_apply_pair does."""
    r.rope3d_testing_na3d_kernel(which)
    r.rope3d_testing_na3d_per_cta(per_cta)
    B, T, H, W, heads, split, kernel = 1, 3, 10, 13, 2, (32, 48, 48), (3, 5, 5)
    shp = (B, T * H * W, heads, 128)
    n = int(np.prod(shp))
    q, k, v = (bf16(synthetic.normal(n, 1.0, 301, i, "bf16")).reshape(shp).to(DEV) for i in range(3))
    tabs = r.rope3d_build_tables(T, H, W, split)
    fused = r.rope3d_na3d(q, k, v, tabs, kernel, apply_rope=True)
    qr, kr = r.rope3d_apply_pair(q, k, tabs)
    unfused = r.rope3d_na3d(qr, kr, v, tabs, kernel, apply_rope=False)
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int16), unfused.view(torch.int16))
    tabs.close()


def test_fused_scratch_is_stream_ordered():
    """rope3d_na3d with the RoPE takes its K scratch from the library's pool
    in stream order: calls queued on two streams, one held back by a spin
    kernel, both give the unfused bits; rope3d_cache_clear then returns the
    pool's memory."""
    B, T, H, W, heads, split, kernel = 1, 4, 16, 24, 2, (32, 48, 48), (3, 7, 7)
    shp = (B, T * H * W, heads, 128)
    n = int(np.prod(shp))
    q, k, v = (bf16(synthetic.normal(n, 1.0, 307, i, "bf16")).reshape(shp).to(DEV) for i in range(3))
    tabs = r.rope3d_build_tables(T, H, W, split)
    qr, kr = r.rope3d_apply_pair(q, k, tabs)
    want = r.rope3d_na3d(qr, kr, v, tabs, kernel, apply_rope=False)
    outs = [torch.empty_like(q) for _ in range(4)]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        torch.cuda._sleep(int(0.2 * 2.0e9))
    for i in range(4):
        r.rope3d_na3d(q, k, v, tabs, kernel, outs[i], stream=s1 if i % 2 == 0 else s2)
    s1.synchronize()
    s2.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), want.view(torch.int16))
    r.rope3d_cache_clear()
    again = r.rope3d_na3d(q, k, v, tabs, kernel)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), want.view(torch.int16))
    tabs.close()


@pytest.mark.parametrize("which", KERNELS)
@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[2]}" for c in CASES])
def test_rotate_once_equals_unfused_bitwise(case, which):
    """K rotated once beforehand and Q in the attention prologue: the unfused
    pair's output bits, and k_rot is rope3d_apply_pair's K_out; the same with
    K rotated in place (k_rot = k)."""
    r.rope3d_testing_na3d_kernel(which)
    (B, T, H, W, heads), split, kernel = case
    shp = (B, T * H * W, heads, 128)
    n = int(np.prod(shp))
    q, k, v = (bf16(synthetic.normal(n, 1.0, 306, i, "bf16")).reshape(shp).to(DEV) for i in range(3))
    tabs = r.rope3d_build_tables(T, H, W, split)
    qr, kr = r.rope3d_apply_pair(q, k, tabs)
    unfused = r.rope3d_na3d(qr, kr, v, tabs, kernel, apply_rope=False)
    out, k_rot = r.rope3d_na3d_rotate_once(q, k, v, tabs, kernel)
    kk = k.clone()
    out2, k_rot2 = r.rope3d_na3d_rotate_once(q, kk, v, tabs, kernel, k_rot=kk)
    torch.cuda.synchronize()
    assert k_rot2 is kk
    for a, b in ((out, unfused), (k_rot, kr), (out2, unfused), (kk, kr)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    tabs.close()


@pytest.mark.parametrize("cap", [1, 176, 4096])
def test_rotate_once_split_k_pass(cap):
    """The K pass cut into launches of whole tokens (1 token, 5 tokens, 128
    tokens per launch, across the batch boundary): the same bits as one
    launch."""
    B, T, H, W, heads, split, kernel = 2, 3, 10, 13, 2, (32, 48, 48), (3, 5, 5)
    shp = (B, T * H * W, heads, 128)
    n = int(np.prod(shp))
    q, k, v = (bf16(synthetic.normal(n, 1.0, 307, i, "bf16")).reshape(shp).to(DEV) for i in range(3))
    tabs = r.rope3d_build_tables(T, H, W, split)
    one, k_one = r.rope3d_na3d_rotate_once(q, k, v, tabs, kernel)
    try:
        r.rope3d_testing_max_units_per_launch(cap)
        split_out, k_split = r.rope3d_na3d_rotate_once(q, k, v, tabs, kernel)
        torch.cuda.synchronize()
    finally:
        r.rope3d_testing_max_units_per_launch(0)
    assert torch.equal(split_out.view(torch.int16), one.view(torch.int16))
    assert torch.equal(k_split.view(torch.int16), k_one.view(torch.int16))
    tabs.close()


def test_rotate_once_rejections():
    B, T, H, W, heads = 1, 3, 8, 8, 1
    tabs = r.rope3d_build_tables(T, H, W, (32, 48, 48))
    shp = (B, T * H * W, heads, 128)
    n = int(np.prod(shp))
    q, k, v = (torch.zeros(shp, dtype=torch.bfloat16, device=DEV) for _ in range(3))
    out = torch.empty_like(q)
    for k_rot in (q, v, out):
        with pytest.raises(r.Rope3dError) as e:
            r.rope3d_na3d_rotate_once(q, k, v, tabs, (3, 3, 3), out=out, k_rot=k_rot)
        assert e.value.name == "ERR_ALIAS"
    flat = torch.empty(n + 8, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_na3d_rotate_once(q, k, v, tabs, (3, 3, 3), out=out, k_rot=flat[1:n + 1].view(shp))
    assert e.value.name == "ERR_ALIGN"
    # K rotated in place while Q is read from the same memory
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_na3d_rotate_once(k, k, v, tabs, (3, 3, 3), out=out, k_rot=k)
    assert e.value.name == "ERR_ALIAS"
    # k_rot overlapping k without being k (one token further on)
    kbig = torch.zeros(n + 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_na3d_rotate_once(q, kbig[:n].view(shp), v, tabs, (3, 3, 3), out=out,
                                  k_rot=kbig[128:].view(shp))
    assert e.value.name == "ERR_ALIAS"
    tabs.close()


@pytest.mark.parametrize("W, kw, want", [(112, 105, 1), (130, 113, 2)], ids=["rows112-tc", "rows120-mma"])
def test_default_kernel_by_region_row_width(W, kw, want):
    """The default attention is the tensor-core kernel while a region row,
    min(W, k_w + 7) keys, fits its 112-key chunk (here exactly: one region
    row a chunk), and the warp-MMA kernel beyond; both within the bound of
    the oracle, with the RoPE."""
    r.rope3d_testing_na3d_kernel(0)
    B, T, H, heads, split, kernel = 1, 2, 5, 1, (32, 48, 48), (1, 3, kw)
    shape6 = (B, T, H, W, heads, 128)
    n = int(np.prod(shape6))
    q_np, k_np, v_np = (synthetic.normal(n, 1.0, 308, i, "bf16") for i in range(3))
    shp = (B, T * H * W, heads, 128)
    q, k, v = (bf16(a).reshape(shp).to(DEV) for a in (q_np, k_np, v_np))
    tabs = r.rope3d_build_tables(T, H, W, split)
    out = r.rope3d_na3d(q, k, v, tabs, kernel)
    torch.cuda.synchronize()
    assert r.rope3d_testing_na3d_last_kernel() == want
    got = to_f64(out).reshape(shape6)
    otabs = oracle.tables(T, H, W, split)
    ref = oracle.rope_na3d(q_np, k_np, v_np, shape6, split, otabs, kernel)
    to64 = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)  # noqa: E731
    qr = oracle.rope3d(q_np, shape6, split, otabs)
    kr = oracle.rope3d(k_np, shape6, split, otabs)
    absv = oracle.na3d(to64(qr), to64(kr), np.abs(to64(v_np)), shape6, kernel)
    bound = 2.0 ** -7 * absv + 2.0 ** -8 * np.abs(ref) + 1e-6
    err = np.abs(got - ref)
    assert np.all(err <= bound), (err.max(), (err / bound).max())
    tabs.close()


def test_single_key_window_returns_v():
    B, T, H, W, heads = 1, 2, 9, 10, 3
    shp = (B, T * H * W, heads, 128)
    n = int(np.prod(shp))
    q, k, v = (bf16(synthetic.normal(n, 1.0, 302, i, "bf16")).reshape(shp).to(DEV) for i in range(3))
    tabs = r.rope3d_build_tables(T, H, W, (32, 48, 48))
    out = r.rope3d_na3d(q, k, v, tabs, (1, 1, 1))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), v.view(torch.int16))
    tabs.close()


def test_na3d_rejections():
    B, T, H, W, heads = 1, 3, 8, 8, 1
    tabs = r.rope3d_build_tables(T, H, W, (32, 48, 48))
    shp = (B, T * H * W, heads, 128)
    q = torch.zeros(shp, dtype=torch.bfloat16, device=DEV)
    for kernel, name in [((2, 3, 3), "ERR_SHAPE"), ((5, 3, 3), "ERR_SHAPE"), ((1, 9, 3), "ERR_SHAPE")]:
        with pytest.raises(r.Rope3dError) as e:
            r.rope3d_na3d(q, q, q, tabs, kernel)
        assert e.value.name == name
    with pytest.raises(r.Rope3dError) as e:
        r.rope3d_na3d(q, q, q, tabs, (3, 3, 3), out=q)
    assert e.value.name == "ERR_ALIAS"
    tabs.close()


def _bench_queries(B, T, H, W, heads, count, seed):
    """Corners, edges and centre of the grid, then seeded random queries."""
    g = np.random.Generator(np.random.PCG64(seed))
    fixed = []
    for t in (0, T // 2, T - 1):
        for h in (0, 1, H // 2, H - 2, H - 1):
            for w in (0, 3, W // 2, W - 1):
                fixed.append((0, t, h, w, int(g.integers(heads))))
    rand = [tuple(int(x) for x in (g.integers(B), g.integers(T), g.integers(H), g.integers(W),
                                   g.integers(heads))) for _ in range(count - len(fixed))]
    return fixed + rand


@pytest.mark.parametrize("which", [0, 2])
def test_na3d_full_size_sampled(which):
    """The attention workload bench.py times (1 x 16 x 64 x 64 tokens, 16
    heads x 128, bf16, window 3 x 7 x 7, same seeds), launched as the bench
    launches it (the default kernel, the tensor-core one here; and the
    warp-MMA kernel): 192 sampled queries of the fused kernel against the oracle
    computed one query at a time, and the unfused pair and the rotate-once
    form bit-identical to it."""
    B, T, H, W, heads, split, kernel = 1, 16, 64, 64, 16, (32, 48, 48), (3, 7, 7)
    shape6 = (B, T, H, W, heads, 128)
    shp = (B, T * H * W, heads, 128)
    n = int(np.prod(shp))
    bits = [synthetic.normal(n, 1.0, 12, i, "bf16") for i in range(3)]
    q, k, v = (bf16(a).reshape(shp).to(DEV) for a in bits)
    tabs = r.rope3d_build_tables(T, H, W, split)
    r.rope3d_testing_na3d_kernel(which)
    fused = r.rope3d_na3d(q, k, v, tabs, kernel)
    qr, kr = r.rope3d_apply_pair(q, k, tabs)
    unfused = r.rope3d_na3d(qr, kr, v, tabs, kernel, apply_rope=False)
    once, k_rot = r.rope3d_na3d_rotate_once(q, k, v, tabs, kernel)
    r.rope3d_testing_na3d_per_cta(True)
    per_cta = r.rope3d_na3d(q, k, v, tabs, kernel)
    r.rope3d_testing_na3d_per_cta(False)
    torch.cuda.synchronize()
    assert r.rope3d_testing_na3d_last_kernel() == (1 if which == 0 else 2)
    assert torch.equal(fused.view(torch.int16), unfused.view(torch.int16))
    assert torch.equal(per_cta.view(torch.int16), unfused.view(torch.int16))
    del per_cta
    assert torch.equal(once.view(torch.int16), unfused.view(torch.int16))
    assert torch.equal(k_rot.view(torch.int16), kr.view(torch.int16))
    del once, k_rot
    queries = _bench_queries(B, T, H, W, heads, 192, 304)
    got_all = fused.view(shape6)
    got = to_f64(torch.stack([got_all[b, t, h, w, e] for b, t, h, w, e in queries]))
    otabs = oracle.tables(T, H, W, split)
    ref, absv = oracle.rope_na3d_at(*bits, shape6, split, otabs, kernel, queries)
    bound = 2.0 ** -7 * absv + 2.0 ** -8 * np.abs(ref) + 1e-6
    err = np.abs(got - ref)
    assert np.all(err <= bound), (err.max(), (err / bound).max())
    tabs.close()


@pytest.mark.parametrize("which", KERNELS)
@pytest.mark.parametrize("path", PATHS)
def test_na3d_large_scores_rescale_often(path, which):
    """Q and K with sigma 3: scores spread over tens of log2 units, so row
    maxima jump by more than 2^8 from chunk to chunk and the running
    reference (and O, l) is rescaled many times; still within the bound."""
    r.rope3d_testing_na3d_kernel(which)
    B, T, H, W, heads, split, kernel = 1, 3, 16, 16, 2, (32, 48, 48), (3, 7, 7)
    shape6 = (B, T, H, W, heads, 128)
    n = int(np.prod(shape6))
    q_np = synthetic.normal(n, 3.0, 305, 0, "bf16")
    k_np = synthetic.normal(n, 3.0, 305, 1, "bf16")
    v_np = synthetic.normal(n, 1.0, 305, 2, "bf16")
    shp = (B, T * H * W, heads, 128)
    q, k, v = (bf16(a).reshape(shp).to(DEV) for a in (q_np, k_np, v_np))
    tabs = r.rope3d_build_tables(T, H, W, split)
    out = attend(path, q, k, v, tabs, kernel)
    torch.cuda.synchronize()
    got = to_f64(out).reshape(shape6)
    otabs = oracle.tables(T, H, W, split)
    ref = oracle.rope_na3d(q_np, k_np, v_np, shape6, split, otabs, kernel)
    to64 = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)  # noqa: E731
    qr = oracle.rope3d(q_np, shape6, split, otabs)
    kr = oracle.rope3d(k_np, shape6, split, otabs)
    # the scores do spread (shown on each token's score with itself): over
    # more than 16 log2 units, twice the rescale threshold
    scores = np.einsum("thwed,thwed->thwe", to64(qr).reshape(shape6)[0], to64(kr).reshape(shape6)[0])
    assert np.ptp(scores) / np.sqrt(128) * 1.4427 > 16
    absv = oracle.na3d(to64(qr), to64(kr), np.abs(to64(v_np)), shape6, kernel)
    bound = 2.0 ** -7 * absv + 2.0 ** -8 * np.abs(ref) + 1e-6
    err = np.abs(got - ref)
    assert np.all(err <= bound), (err.max(), (err / bound).max())
    tabs.close()
