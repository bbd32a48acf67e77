"""The seeded input generator: structure, determinism and bf16 rounding."""
import numpy as np
import torch

from speculative_decoding_verify_lm_gb300 import synth


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 3,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0, 1e-30], np.float32)])
    ours = synth.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_normal_bf16_deterministic_and_thread_independent():
    a = synth.normal_bf16(123, 0, 3000, 64, 0.02, chunk_rows=512, threads=1)
    b = synth.normal_bf16(123, 0, 3000, 64, 0.02, chunk_rows=512, threads=8)
    assert np.array_equal(a, b)
    v = synth.bf16_bits_to_f32(a)
    assert abs(v.std() - 0.02) < 0.001 and abs(v.mean()) < 0.001


def test_random_tree_shape():
    rng = np.random.default_rng(1)
    for _ in range(50):
        parent, dep = synth.random_tree(rng, 60, 8, 10)
        assert len(parent) == 60 and dep.max() == 8
        assert all(parent[i] < i for i in range(60))
        kids = np.bincount(parent + 1, minlength=61)
        assert kids.max() <= 10
        for i in range(60):
            assert dep[i] == 1 + (0 if parent[i] < 0 else dep[parent[i]])
        assert all(dep[i] <= dep[i + 1] for i in range(59))      # breadth-first labels


def _fake_argmax(W, rows):
    # a stand-in target choice (not the method's arithmetic): a hash of the row
    ids = (rows.astype(np.int64).sum(axis=1) * 2654435761) % W.shape[0]
    return ids.astype(np.int32), None


def test_planting_structure():
    wl = synth.small_workload(5, d=32, V=97, kinds=[0, 1, 1, 0], argmax_fn=_fake_argmax, m=8,
                              n_nodes=30, depth=6, branch=5, reject=False)
    g, _ = _fake_argmax(wl.W, wl.hidden)
    for b in range(wl.B):
        r0, n0 = wl.pos_off[b], wl.node_off[b]
        tok = wl.tok[n0:wl.node_off[b + 1]]
        par = wl.parent[n0:wl.node_off[b + 1]]
        path = wl.path_nodes[b]
        cut = wl.cut[b]
        for depth, node in enumerate(path, start=1):
            prow = r0 if par[node] < 0 else r0 + 1 + par[node]
            if depth <= cut:
                assert tok[node] == g[prow]
            elif depth == cut + 1:
                assert tok[node] != g[prow]
        if wl.kind[b] == 1:
            on_path = set(path)
            for i in range(len(tok)):
                prow = r0 if par[i] < 0 else r0 + 1 + par[i]
                if i not in on_path:
                    assert tok[i] != g[prow]
            for p in set(par.tolist()):
                sib = tok[par == p]
                assert len(set(sib.tolist())) == len(sib)


def test_config_shapes():
    sizes = {}
    for i, cfg in enumerate(synth.CONFIGS):
        kinds, parents, paths, cuts, pos_off, node_off = synth._structure(cfg, synth.seed_of(i), cfg.B)
        sizes[cfg.name] = int(pos_off[-1])
        assert len(kinds) == cfg.B
        if cfg.kind == "mixed":
            assert kinds.sum() == cfg.B // 2
        assert all(0 <= c <= (cfg.K if k == 0 else cfg.depth) for c, k in zip(cuts, kinds))
    assert sizes == {"tiny_chain_b1": 17, "qwen3_4b_dflash_chain_b1": 17, "qwen3_4b_eagle3_tree_b1": 61,
                     "qwen3_4b_mixed_b32": 1248, "qwen3_4b_tree_b256": 15616}


def test_geometric_cut_mean():
    rng = np.random.default_rng(2)
    cuts = np.minimum(rng.geometric(0.25, 200000) - 1, 16)
    assert abs(cuts.mean() - (3 - 0.75 ** 17 * 4)) < 0.05
