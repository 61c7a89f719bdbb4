"""GPU parity: tv_tree_attention against the oracle (fp64).

Tolerances: 1e-4 max-abs for fp32 inputs (CUDA-core kernel), 2e-2 max-abs for bf16
inputs (tensor-core kernel: bf16 operands, fp32 accumulation and softmax, P rounded to
bf16 for the second product).  Sizes span several 128-row tiles, several 64-key KV tiles
with ragged tails, one and several KV splits, and the full workload shapes (sampled
rows where the oracle would be slow)."""
import math

import numpy as np
import pytest

import synth
import synth.workloads as W
from oracle import attention, selection

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import tree_speculative_decoding_masked_gb300 as tv  # noqa: E402
from gpu_util import dev, host, i32, to_dev  # noqa: E402


def _run(q, k, v, par, P, bf16, stride_pad=0, pad_value=None):
    qd = to_dev(q, bf16)
    if stride_pad:
        B, H, L, D = k.shape
        kp = np.zeros((B, H, L + stride_pad, D), dtype=np.float32)
        vp = np.zeros_like(kp)
        kp[:, :, :L] = k
        vp[:, :, :L] = v
        kd, vd = to_dev(kp, bf16), to_dev(vp, bf16)
        if pad_value is not None:
            kd[:, :, L:] = pad_value
            vd[:, :, L:] = pad_value
    else:
        kd, vd = to_dev(k, bf16), to_dev(v, bf16)
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    out = tv.tree_attention(qd, kd, vd, i32(par), P, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return host(out)


def _check_all(q, k, v, par, P, bf16, **kw):
    got = _run(q, k, v, par, P, bf16, **kw)
    ref = attention.tree_attention(q, k, v, par, P)
    err = float(np.max(np.abs(got - ref)))
    assert np.isfinite(got).all()
    assert err < (2e-2 if bf16 else 1e-4), err
    return err


def test_tiny_fp32_workload():
    cfg = W.WORKLOADS["tiny_fp32"]
    g = synth.rng(cfg["seed"])
    par, _ = W.trees(g, cfg["B"], cfg["N"], cfg["depth_cap"], cfg["V"])
    q, k, v = W.qkv_host(g, cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["P"], cfg["N"], False)
    _check_all(q, k, v, par, cfg["P"], False)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("shape", [
    # B, Hq, Hkv, D, P, N, depth cap
    (2, 8, 2, 128, 300, 37, 5),     # one split, ragged tiles
    (1, 8, 2, 128, 1000, 70, 8),    # several splits, two row tiles
    (2, 4, 4, 64, 130, 129, 16),    # G = 1, D = 64, 2 row tiles
    (1, 16, 2, 128, 200, 33, 4),    # G = 8 (16 nodes per row tile)
    (1, 6, 2, 64, 77, 45, 3),       # G = 3 (40-node row tiles, 8 padding rows)
    (1, 4, 1, 128, 0, 64, 6),       # empty prefix: tree keys only
    (1, 4, 1, 128, 64, 16, 2),      # prefix ends on a tile boundary
])
def test_shapes(bf16, shape):
    B, Hq, Hkv, D, P, N, cap = shape
    g = synth.rng(sum(shape) + int(bf16))
    par, _ = W.trees(g, B, N, cap, 100)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, bf16)
    _check_all(q, k, v, par, P, bf16)


@pytest.mark.parametrize("bf16", [False, True])
def test_chain_tree_is_causal_attention(bf16):
    B, Hq, Hkv, D, P, N = 1, 8, 2, 128, 500, 40
    g = synth.rng(31)
    par = synth.chain_parents(N)[None]
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, bf16)
    got = _run(q, k, v, par, P, bf16)
    for h in range(Hq):
        ref = attention.causal_attention(q[0, h], k[0, h // 4, :P + N], v[0, h // 4, :P + N], 1 / math.sqrt(D))
        assert np.max(np.abs(got[0, h] - ref)) < (2e-2 if bf16 else 1e-4)


@pytest.mark.parametrize("bf16", [False, True])
def test_star_tree(bf16):
    B, Hq, Hkv, D, P, N = 1, 4, 1, 64, 100, 100
    g = synth.rng(32)
    par = synth.star_parents(N)[None]
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, bf16)
    _check_all(q, k, v, par, P, bf16)


def test_cache_padding_rows_never_read():
    # rows between P + N and the cache stride hold NaN; the output must not see them
    B, Hq, Hkv, D, P, N = 1, 8, 2, 128, 190, 30
    g = synth.rng(33)
    par, _ = W.trees(g, B, N, 4, 100)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, True)
    got = _run(q, k, v, par, P, True, stride_pad=50, pad_value=float("nan"))
    ref = attention.tree_attention(q, k, v, par, P)
    assert np.isfinite(got).all() and np.max(np.abs(got - ref)) < 2e-2


def test_large_scores_rescale_path():
    # scores that grow along the key axis force the running-max rescale of O
    B, Hq, Hkv, D, P, N = 1, 4, 1, 128, 1000, 32
    g = synth.rng(34)
    par, _ = W.trees(g, B, N, 4, 100)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, False)
    ramp = np.linspace(0.0, 6.0, P + N, dtype=np.float32)[None, None, :, None]
    k = synth.round_to_bf16((k * 0.2 + ramp * np.sign(q.mean(axis=(0, 1, 2)))[None, None, None, :]).astype(np.float32))
    q = synth.round_to_bf16(q)
    v = synth.round_to_bf16(v)
    _check_all(q, k, v, par, P, True)


def test_qwen3_4b_layer_workload_all_rows():
    cfg = W.WORKLOADS["qwen3_4b_layer"]
    g = synth.rng(cfg["seed"])
    marg, ptok = W.pools(g, 1, cfg["pool_d"], cfg["pool_k"], cfg["V"])
    par = selection.select_subtree(marg[0], ptok[0], cfg["N"], 11)["parent"][None]
    q, k, v = W.qkv_host(g, 1, cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["P"], cfg["N"], True)
    _check_all(q, k, v, par, cfg["P"], True)


def _tree_dominated(qd, kd, P, N, seed, gamma=13.0):
    """Add gamma * u (u a seeded unit vector) to every query and to the tree's key rows
    P..P+N-1: a node's tree keys then score about gamma^2 / sqrt(D) ~ 15 above the
    prefix keys, more than ln(P) + a margin, so the ancestors carry most of the softmax
    mass and a wrong ancestor set or a wrong tile boundary at P moves the output by O(1)."""
    D = qd.shape[-1]
    gen = torch.Generator(device=qd.device)
    gen.manual_seed(int(seed))
    u = torch.randn(D, generator=gen, device=qd.device, dtype=torch.float32)
    u /= u.norm()
    qd = (qd.float() + gamma * u).to(qd.dtype)
    kd = kd.clone()
    kd[:, :, P:P + N] = (kd[:, :, P:P + N].float() + gamma * u).to(kd.dtype)
    return qd, kd


def _sampled_rows(name, n_rows, seed_extra=0, tree_dominated=False):
    cfg = W.WORKLOADS[name]
    B, Hq, Hkv, D, P = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["P"]
    N = cfg.get("N", 1024)
    g = synth.rng(cfg["seed"] + seed_extra)
    par, _ = W.trees(g, B, N, cfg.get("depth_cap", 16), 100)
    qd = W.device_normal((B, Hq, N, D), 1.0, cfg["seed"] + 1, torch.bfloat16, dev())
    kd = W.device_normal((B, Hkv, P + N, D), 1.0, cfg["seed"] + 2, torch.bfloat16, dev())
    vd = W.device_normal((B, Hkv, P + N, D), 1.0, cfg["seed"] + 3, torch.bfloat16, dev())
    if tree_dominated:
        qd, kd = _tree_dominated(qd, kd, P, N, cfg["seed"] + 4)
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    out = tv.tree_attention(qd, kd, vd, i32(par), P, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    G = Hq // Hkv
    rows = [(int(g.integers(B)), int(g.integers(Hq)), int(g.integers(N))) for _ in range(n_rows)]
    rows += [(0, 0, i) for i in range(0, N, max(1, N // 64))]  # a spread of nodes of one head
    rows += [(B - 1, Hq - 1, N - 1)]
    worst = 0.0
    cache = {}
    tree_mass = []
    for b, h, i in rows:
        key = (b, h // G)
        if key not in cache:
            cache[key] = (kd[b, h // G].float().cpu().numpy()[None, None], vd[b, h // G].float().cpu().numpy()[None, None])
        kk, vv = cache[key]
        qq = qd[b, h].float().cpu().numpy()[None, None]
        ref = attention.per_node_bruteforce(qq, kk, vv, par[b:b + 1], P, 0, 0, i)
        got = out[b, h, i].float().cpu().numpy()
        worst = max(worst, float(np.max(np.abs(got - ref))))
        if tree_dominated:  # share of the softmax mass on the node's tree keys (test power)
            path = [P + t for t in _root_path(par[b], i)]
            sc = (kk[0, 0, :P + N].astype(np.float64) @ qq[0, 0, i].astype(np.float64)) / math.sqrt(D)
            w = np.exp(sc[:P] - sc[path].max())
            tree_mass.append(np.exp(sc[path] - sc[path].max()).sum() / (w.sum() + np.exp(sc[path] - sc[path].max()).sum()))
    assert worst < 2e-2, worst
    if tree_dominated:
        assert np.median(tree_mass) > 0.9, np.median(tree_mass)


def test_long_context_workload_sampled():
    _sampled_rows("long_context", 48)


def test_sampling_workload_sampled():
    _sampled_rows("sampling", 48)


def test_budget_sweep_1024_nodes_sampled():
    _sampled_rows("budget_sweep", 48)


def _root_path(parent, i):
    path = []
    while i >= 0:
        path.append(int(i))
        i = int(parent[i])
    return path[::-1]


@pytest.mark.parametrize("name", ["long_context", "budget_sweep"])
def test_full_size_tree_dominated(name):
    # prefix 32768 / 128-node trees and prefix 4096 / 1024-node trees with the softmax
    # mass on each node's ancestors: the mask and the KV tile and split boundaries at P
    # decide the output at full size
    _sampled_rows(name, 48, seed_extra=9, tree_dominated=True)


def test_bad_tree_flagged():
    B, Hq, Hkv, D, P, N = 1, 8, 2, 128, 64, 8
    g = synth.rng(35)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, True)
    par = np.array([[-1, 0, 1, 5, 2, 3, 4, 5]], dtype=np.int32)
    for bf16 in (True, False):
        st = torch.zeros(1, dtype=torch.int32, device=dev())
        tv.tree_attention(to_dev(q, bf16), to_dev(k, bf16), to_dev(v, bf16), i32(par), P, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) & tv.TV_DEV_BAD_TREE


@pytest.fixture(params=[1, 2, 3, 4, 5],
                ids=["one_tile_per_cta", "paired_tiles", "paired_tiles_64key_double_s", "persistent_grid", "sm_pairs"])
def variant(request):
    tv.set_attention_variant(request.param)
    yield request.param
    tv.set_attention_variant(0)


@pytest.mark.parametrize("shape", [
    # B, Hq, Hkv, D, P, N, depth cap
    (1, 8, 2, 128, 1000, 70, 8),    # three row tiles: one full pair and a pair with no second tile
    (1, 8, 2, 128, 96, 64, 6),      # the pair's second tile needs one KV tile more than the first
    (2, 4, 4, 64, 130, 129, 16),    # G = 1, D = 64, two row tiles
    (1, 6, 2, 64, 77, 45, 3),       # G = 3, padding rows in every tile
    (1, 4, 1, 128, 0, 300, 16),     # empty prefix, three row tiles of tree keys only
    (2, 32, 8, 128, 2048, 64, 8),   # the qwen3 layer shape, two sequences (KV splits in clusters)
    (1, 4, 1, 128, 5000, 96, 12),   # many KV tiles per split, the last split shorter
])
def test_shapes_both_variants(variant, shape):
    B, Hq, Hkv, D, P, N, cap = shape
    g = synth.rng(sum(shape) + 7)
    par, _ = W.trees(g, B, N, cap, 100)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, True)
    _check_all(q, k, v, par, P, True)


def test_rescale_path_both_variants(variant):
    # scores growing along the key axis force O rescales in either kernel
    B, Hq, Hkv, D, P, N = 1, 4, 1, 128, 3000, 200
    g = synth.rng(36)
    par, _ = W.trees(g, B, N, 8, 100)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, False)
    ramp = np.linspace(0.0, 6.0, P + N, dtype=np.float32)[None, None, :, None]
    k = synth.round_to_bf16((k * 0.2 + ramp * np.sign(q.mean(axis=(0, 1, 2)))[None, None, None, :]).astype(np.float32))
    _check_all(synth.round_to_bf16(q), k, synth.round_to_bf16(v), par, P, True)


def test_chain_and_star_both_variants(variant):
    B, Hq, Hkv, D, P, N = 1, 8, 2, 128, 700, 100
    g = synth.rng(37)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, True)
    got = _run(q, k, v, synth.chain_parents(N)[None], P, True)
    for h in range(Hq):
        ref = attention.causal_attention(q[0, h], k[0, h // 4, :P + N], v[0, h // 4, :P + N], 1 / math.sqrt(D))
        assert np.max(np.abs(got[0, h] - ref)) < 2e-2
    _check_all(q, k, v, synth.star_parents(N)[None], P, True)


def test_long_context_workload_sampled_one_tile_per_cta():
    tv.set_attention_variant(1)
    try:
        _sampled_rows("long_context", 24, seed_extra=5)
    finally:
        tv.set_attention_variant(0)


@pytest.mark.parametrize("name", ["long_context", "sampling", "budget_sweep"])
def test_workloads_sampled_64key_double_s(name):
    tv.set_attention_variant(3)
    try:
        _sampled_rows(name, 24, seed_extra=6)
    finally:
        tv.set_attention_variant(0)


@pytest.mark.parametrize("name", ["long_context", "sampling", "budget_sweep"])
def test_workloads_sampled_sm_pairs(name):
    # every product of the paired 64-key kernel as one M = 256 MMA over the row tiles of
    # two CTAs (an SM pair), each CTA holding half of every K and V tile
    tv.set_attention_variant(5)
    try:
        cfg = W.WORKLOADS[name]
        assert tv.tree_attention_plan(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["P"], cfg.get("N", 1024),
                                      torch.bfloat16) == (5, 1)
        _sampled_rows(name, 24, seed_extra=7)
    finally:
        tv.set_attention_variant(0)


@pytest.mark.parametrize("name", ["long_context", "budget_sweep"])
def test_full_size_tree_dominated_sm_pairs(name):
    tv.set_attention_variant(5)
    try:
        _sampled_rows(name, 32, seed_extra=10, tree_dominated=True)
    finally:
        tv.set_attention_variant(0)


@pytest.mark.parametrize("n_active", [128, 100, 50, 20])
def test_sm_pairs_ragged_rows(n_active):
    # SM pairs over ragged rows: with 50 active nodes sequence 1's second CTA of the pair
    # has no active row but still holds half of every product; with 20 only the first
    # row tile of the first CTA is active
    B, Hq, Hkv, D, P, N = 2, 4, 1, 128, 2000, 128
    g = synth.rng(61 + n_active)
    par, _ = W.trees(g, B, N, 9, 100)
    par[1, n_active:] = -1
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, True)
    out = torch.full((B, Hq, N, D), 7.0, dtype=torch.bfloat16, device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    tv.set_attention_variant(5)
    try:
        assert tv.tree_attention_plan(B, Hq, Hkv, D, P, N, torch.bfloat16) == (5, 1)
        tv.tree_attention(to_dev(q, True), to_dev(k, True), to_dev(v, True), i32(par), P, out=out, dev_status=st)
        torch.cuda.synchronize()
    finally:
        tv.set_attention_variant(0)
    assert int(st.item()) == 0
    got = host(out)
    ref = attention.tree_attention(q, k, v, par, P)
    assert np.max(np.abs(got[0] - ref[0])) < 2e-2
    assert np.max(np.abs(got[1, :, :n_active] - ref[1, :, :n_active])) < 2e-2
    assert (got[1, :, n_active:] == 7.0).all()


@pytest.mark.parametrize("name", ["long_context", "sampling", "budget_sweep"])
def test_workloads_sampled_persistent_grid(name):
    tv.set_attention_variant(4)
    try:
        _sampled_rows(name, 24, seed_extra=7)
    finally:
        tv.set_attention_variant(0)


@pytest.mark.parametrize("share", [16, 40, 0])
def test_persistent_grid_many_pieces_per_cta(share):
    # four tile pairs per (sequence, KV head) of 1..4 64-key steps, 80 steps in all: on
    # 16 SMs a CTA's range of 5 steps holds up to seven pieces (whole units between a
    # partial one at each end), on 40 up to four, on the whole device (80 CTAs) one step
    # each, a 4-step unit merged from four CTAs; every cut matches the oracle
    B, Hq, Hkv, D, P, N = 4, 8, 2, 64, 0, 256
    g = synth.rng(41 + share)
    par, _ = W.trees(g, B, N, 9, 100)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, True)
    tv.set_attention_variant(4)
    tv.set_sm_partition(0, share)
    try:
        assert tv.tree_attention_plan(B, Hq, Hkv, D, P, N, torch.bfloat16) == (4, 1)
        _check_all(q, k, v, par, P, True)
    finally:
        tv.set_attention_variant(0)
        tv.set_sm_partition(0, 0)


def test_persistent_grid_without_workspace_runs_paired_kernel():
    # a workspace smaller than the query: the same result through the unsplit paired kernel
    B, Hq, Hkv, D, P, N = 2, 8, 2, 128, 3000, 64
    g = synth.rng(44)
    par, _ = W.trees(g, B, N, 6, 100)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, True)
    tv.set_attention_variant(4)
    try:
        assert tv.tree_attention_workspace_size(B, Hq, Hkv, D, P, N, torch.bfloat16) > 0
        st = torch.zeros(1, dtype=torch.int32, device=dev())
        out = tv.tree_attention(to_dev(q, True), to_dev(k, True), to_dev(v, True), i32(par), P,
                                workspace=torch.zeros(256, dtype=torch.uint8, device=dev()), dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref = attention.tree_attention(q, k, v, par, P)
        assert np.max(np.abs(host(out) - ref)) < 2e-2
    finally:
        tv.set_attention_variant(0)


@pytest.mark.parametrize("n_active,D", [(128, 128), (100, 128), (50, 128), (100, 64)])
def test_kv_multicast_tile_pairs(n_active, D):
    # a prefix of at least 64 N keys: the paired 64-key kernel runs its tile pairs in
    # clusters of two that share each K/V tile (each CTA loads half of its rows into both
    # rings).  Ragged rows: with 50 active nodes sequence 1's second tile pair has no
    # active row and only streams the tiles its partner needs; with 100 the two pairs'
    # key ranges differ.
    B, Hq, Hkv, P, N = 2, 4, 1, 8192, 128
    g = synth.rng(45 + n_active + D)
    par, _ = W.trees(g, B, N, 9, 100)
    par[1, n_active:] = -1
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, True)
    out = torch.full((B, Hq, N, D), 7.0, dtype=torch.bfloat16, device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    tv.set_attention_variant(3)  # this small grid would otherwise run split single tiles
    tv.set_attention_splits(1)
    try:
        assert tv.tree_attention_plan(B, Hq, Hkv, D, P, N, torch.bfloat16) == (3, 1)
        tv.tree_attention(to_dev(q, True), to_dev(k, True), to_dev(v, True), i32(par), P, out=out, dev_status=st)
        torch.cuda.synchronize()
    finally:
        tv.set_attention_variant(0)
        tv.set_attention_splits(0)
    assert int(st.item()) == 0
    got = host(out)
    ref = attention.tree_attention(q, k, v, par, P)
    assert np.max(np.abs(got[0] - ref[0])) < 2e-2
    assert np.max(np.abs(got[1, :, :n_active] - ref[1, :, :n_active])) < 2e-2
    assert (got[1, :, n_active:] == 7.0).all()


@pytest.mark.parametrize("splits", [1, 3, 8])
def test_forced_splits_both_variants(variant, splits):
    # every split count merges to the same result, including more splits than a short
    # KV range has tiles (the last CTAs of a cluster then own no keys)
    B, Hq, Hkv, D, P, N = 2, 8, 2, 128, 600, 90
    g = synth.rng(38 + splits)
    par, _ = W.trees(g, B, N, 7, 100)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, True)
    tv.set_attention_splits(splits)
    try:
        _check_all(q, k, v, par, P, True)
    finally:
        tv.set_attention_splits(0)


def test_fp32_many_rows_four_rows_per_warp():
    # more than 4096 query rows: the CUDA-core kernel gives each warp four rows (small
    # problems get one row per warp); fp32 within 1e-4
    B, Hq, Hkv, D, P, N = 2, 32, 8, 64, 100, 80
    g = synth.rng(39)
    par, _ = W.trees(g, B, N, 6, 100)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, False)
    _check_all(q, k, v, par, P, False)


def test_attention_plan_query_and_overrides():
    # the plan query names a tensor-core kernel for bf16 tile shapes and the CUDA-core one
    # for fp32; forced variants and split counts are what the query then reports
    assert tv.tree_attention_plan(1, 4, 1, 64, 128, 16, torch.float32) == (0, 1)
    k, s = tv.tree_attention_plan(8, 32, 8, 128, 32768, 128, torch.bfloat16)
    assert k in (1, 3, 4) and 1 <= s <= 8
    try:
        tv.set_attention_variant(1)
        tv.set_attention_splits(3)
        assert tv.tree_attention_plan(2, 8, 2, 128, 1000, 70, torch.bfloat16) == (1, 3)
        tv.set_attention_variant(2)
        tv.set_attention_splits(0)
        assert tv.tree_attention_plan(2, 8, 2, 128, 1000, 70, torch.bfloat16)[0] == 2
        tv.set_attention_variant(3)
        assert tv.tree_attention_plan(2, 8, 2, 128, 1000, 70, torch.bfloat16)[0] == 3
        tv.set_attention_variant(4)
        assert tv.tree_attention_plan(2, 8, 2, 128, 1000, 70, torch.bfloat16) == (4, 1)
        tv.set_attention_splits(3)  # a forced split count: the paired kernel with splits
        assert tv.tree_attention_plan(2, 8, 2, 128, 1000, 70, torch.bfloat16) == (3, 3)
        tv.set_attention_variant(5)  # SM pairs: D = 128, no splits, tile pairs in twos
        assert tv.tree_attention_plan(2, 8, 2, 128, 1000, 70, torch.bfloat16) == (3, 3)
        tv.set_attention_splits(0)
        assert tv.tree_attention_plan(2, 8, 2, 128, 1000, 70, torch.bfloat16) == (5, 1)
        assert tv.tree_attention_plan(2, 8, 2, 64, 1000, 70, torch.bfloat16)[0] == 3
        assert tv.tree_attention_plan(2, 8, 2, 128, 96, 64, torch.bfloat16)[0] == 3  # one tile pair
    finally:
        tv.set_attention_variant(0)
        tv.set_attention_splits(0)
    with pytest.raises(Exception):
        tv.set_attention_splits(9)
