"""Runs a fixed set of small verify-round calls through one build of the
library and saves every output: `python tests/_checked_cases.py LIB OUT.npz`.
test_gpu_checked_build.py runs it once with libglance.so and once with the
bounds-checked libglance_check.so and compares the two. Inputs are seeded."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import tree_verified_block_gb300._binding as b  # noqa: E402

b.LIB_PATH = sys.argv[1]

import torch  # noqa: E402

import tree_verified_block_gb300 as g  # noqa: E402
import workloads as W  # noqa: E402


def bf16(bits, dev):
    return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)


def main(out_path):
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    res = {}
    L, V, Hq, Hkv, D, d = 15, 4096, 8, 2, 128, 256
    gen = W.rng(21)

    # one request: build, attention (cooperative split merge), LM head (one
    # CTA per column block), walk + commit
    N, T = 31, 700
    rows = N + 1
    x = torch.from_numpy(W.draft_logits_planted(L, V, seed=5)).to(dev)
    tree = g.Tree(N, L, dev)
    t_len = torch.tensor([T], dtype=torch.int32, device=dev)
    g.build_tree(x, N, torch.tensor([3], dtype=torch.int32, device=dev), t_len, tree,
                 g.workspace(g.build_tree_workspace_bytes(L, V, N), dev))
    for k, v in tree.to_host().items():
        res[f"tree_{k}"] = v
    K = bf16(W.normal_bf16(gen, (Hkv, T + rows + 8, D)), dev)
    Vc = bf16(W.normal_bf16(gen, (Hkv, T + rows + 8, D)), dev)
    layer = g.KVLayer(K, Vc, t_len)
    q = bf16(W.normal_bf16(gen, (rows, Hq, D)), dev)
    out = torch.empty_like(q)
    g.tree_attention(q, layer, tree, D ** -0.5, out,
                     g.workspace(g.tree_attention_workspace_bytes(rows, Hq, layer), dev))
    res["attn"] = out.view(torch.int16).cpu().numpy()
    qf, Kf, Vf = q.float(), K.float(), Vc.float()
    layer_f = g.KVLayer(Kf, Vf, t_len)
    out_f = torch.empty_like(qf)
    g.tree_attention(qf, layer_f, tree, D ** -0.5, out_f,
                     g.workspace(g.tree_attention_workspace_bytes(rows, Hq, layer_f), dev))
    res["attn_f32"] = out_f.cpu().numpy()
    h = bf16(W.normal_bf16(gen, (rows, d)), dev)
    Wm = bf16(W.normal_bf16(gen, (d, V), std=0.02), dev)
    am = torch.empty(rows, dtype=torch.int32, device=dev)
    gap = torch.empty(rows, dtype=torch.float32, device=dev)
    g.lmhead_argmax(h, Wm, am, gap, None, g.workspace(g.lmhead_argmax_workspace_bytes(rows, d, V, torch.bfloat16), dev))
    res["argmax"], res["gap"] = am.cpu().numpy(), gap.cpu().numpy()
    n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
    acc_tok = torch.zeros(L, dtype=torch.int32, device=dev)
    new_root = torch.zeros(1, dtype=torch.int32, device=dev)
    g.accept_commit(tree, am, [layer], n_acc, acc_tok, new_root,
                    g.workspace(g.accept_commit_workspace_bytes(1), dev))
    res["commit"] = np.concatenate([n_acc.cpu().numpy(), acc_tok.cpu().numpy(), new_root.cpu().numpy(),
                                    t_len.cpu().numpy()])
    res["cache_k"] = K.view(torch.int16)[:, T:T + rows].cpu().numpy()

    # a ragged batch: batched build, attention in ticket mode, the LM head's
    # CTA-pair kernel (M = 192 > 128), batched commit, tree-row K/V scatter
    B, N2 = 3, 63
    rows2 = N2 + 1
    Ts = [100, 1500, 4000]
    xb = torch.from_numpy(np.stack([W.draft_logits_planted(L, V, seed=40 + r) for r in range(B)])).to(dev)
    trees = [g.Tree(N2, L, dev) for _ in range(B)]
    t_lens = torch.tensor(Ts, dtype=torch.int32, device=dev)
    g.build_tree_batched(xb, N2, torch.tensor([7, 8, 9], dtype=torch.int32, device=dev), t_lens, trees,
                         g.workspace(g.build_tree_batched_workspace_bytes(B, L, V, N2), dev))
    for r in range(B):
        for k, v in trees[r].to_host().items():
            res[f"btree{r}_{k}"] = v
    kvs = []
    for r in range(B):
        kc = bf16(W.normal_bf16(gen, (Hkv, Ts[r] + rows2 + 16, D)), dev)
        vc = bf16(W.normal_bf16(gen, (Hkv, Ts[r] + rows2 + 16, D)), dev)
        kvs.append(g.KVLayer(kc, vc, t_lens[r:r + 1]))
    src = bf16(W.normal_bf16(gen, (1, 2, Hkv, rows2, D)), dev)
    for r in range(B):
        g.kv_write_rows(src, [kvs[r]], rows2)
    qb = bf16(W.normal_bf16(gen, (B, rows2, Hq, D)), dev)
    ob = torch.empty_like(qb)
    g.tree_attention_batched(qb, kvs, trees, D ** -0.5, ob,
                             g.workspace(g.tree_attention_batched_workspace_bytes(rows2, Hq, kvs), dev))
    res["battn"] = ob.view(torch.int16).cpu().numpy()
    M = B * rows2
    hb = bf16(W.normal_bf16(gen, (M, d)), dev)
    amb = torch.empty(M, dtype=torch.int32, device=dev)
    gapb = torch.empty(M, dtype=torch.float32, device=dev)
    g.lmhead_argmax(hb, Wm, amb, gapb, None, g.workspace(g.lmhead_argmax_workspace_bytes(M, d, V, torch.bfloat16), dev))
    res["bargmax"], res["bgap"] = amb.cpu().numpy(), gapb.cpu().numpy()
    n_accb = torch.zeros(B, dtype=torch.int32, device=dev)
    acc_tokb = torch.zeros((B, L), dtype=torch.int32, device=dev)
    new_rootb = torch.zeros(B, dtype=torch.int32, device=dev)
    g.accept_commit_batched(trees, amb.view(B, rows2), [[kvs[r]] for r in range(B)], n_accb, acc_tokb,
                            new_rootb, g.workspace(g.accept_commit_batched_workspace_bytes(B, 1), dev))
    res["bcommit"] = np.concatenate([n_accb.cpu().numpy(), acc_tokb.cpu().numpy().ravel(),
                                     new_rootb.cpu().numpy(), t_lens.cpu().numpy()])

    st = torch.zeros(g.STATUS_WORDS, dtype=torch.int32, device=dev)
    g.get_status(st)
    torch.cuda.synchronize()
    res["status"] = st.cpu().numpy()
    np.savez(out_path, **res)


if __name__ == "__main__":
    main(sys.argv[2])
