"""Block copy on the GPU, and decode attention over block tables that the host
block pool hands out (fork, copy-on-write, cached prefixes), against dense
attention on each sequence's own token list (no block tables involved)."""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("kv,D", [("fp16", 128), ("bf16", 64), ("e5m2", 128), ("int8", 128)])
def test_copy_blocks_bit_exact(dev, kv, D):
    import paged_kv_cache_252_gb300 as pkv
    nb, Hkv = 40, 4
    kc, vc = pkv.alloc_kv_cache(nb, Hkv, D, kv, dev)
    g = torch.Generator(device="cpu").manual_seed(5)
    sc = pkv.alloc_kv_scales(nb, Hkv, dev) if kv == "int8" else None
    for c in (kc, vc) + ((sc,) if sc is not None else ()):
        c.view(torch.uint8).copy_(torch.randint(0, 256, c.view(torch.uint8).shape, generator=g,
                                                dtype=torch.uint8).to(dev))
    k0, v0 = kc.clone(), vc.clone()
    s0 = sc.clone() if sc is not None else None
    perm = torch.randperm(nb, generator=g)
    src, dst = perm[:12].to(torch.int32), perm[12:24].to(torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.copy_blocks(kc, vc, src.to(dev), dst.to(dev), scales=sc, device_status=status)
    torch.cuda.synchronize()
    ek, ev = k0.clone(), v0.clone()
    ek[dst.long().to(dev)] = k0[src.long().to(dev)]
    ev[dst.long().to(dev)] = v0[src.long().to(dev)]
    assert torch.equal(kc.view(torch.uint8), ek.view(torch.uint8))
    assert torch.equal(vc.view(torch.uint8), ev.view(torch.uint8))
    if sc is not None:
        es = s0.clone()
        es[dst.long().to(dev)] = s0[src.long().to(dev)]
        assert torch.equal(sc.view(torch.uint8), es.view(torch.uint8))
    assert int(status.item()) == 0
    # an out-of-range id is skipped and flagged
    bad_src = torch.tensor([nb + 3, int(src[0])], dtype=torch.int32, device=dev)
    bad_dst = torch.tensor([int(dst[0]), -1], dtype=torch.int32, device=dev)
    before = kc.clone()
    pkv.copy_blocks(kc, vc, bad_src, bad_dst, scales=sc, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x2 and torch.equal(kc.view(torch.uint8), before.view(torch.uint8))


def _dense_attention(q, k, v, scale, n):
    """fp64 attention of n query tokens (the last n positions, causal among
    themselves) over one sequence's contiguous K/V [ctx, Hkv, D]; GQA groups."""
    q, k, v = q.double(), k.double(), v.double()
    ctx, Hkv, D = k.shape
    Hq = q.shape[1]
    G = Hq // Hkv
    out = torch.empty(n, Hq, D, dtype=torch.float64)
    for j in range(n):
        lim = ctx - n + j + 1
        for hq in range(Hq):
            s = (k[:lim, hq // G] @ q[j, hq]) * scale
            w = torch.softmax(s, dim=0)
            out[j, hq] = w @ v[:lim, hq // G]
    return out


@pytest.mark.parametrize("kv,Hq,Hkv,n", [("fp16", 32, 8, 1), ("e5m2", 64, 8, 4)])
def test_decode_over_forked_and_cached_sequences(dev, kv, Hq, Hkv, n):
    import paged_kv_cache_252_gb300 as pkv
    D, nb = 128, 64
    scale = 1.0 / math.sqrt(D)
    g = torch.Generator(device="cpu").manual_seed(11)
    pool = pkv.BlockAllocator(nb)
    kc, vc = pkv.alloc_kv_cache(nb, Hkv, D, kv, dev)
    tokens, kv_tok = {}, {}          # sequence -> token ids, per-token (K, V) in fp16

    def write(seq, new_ids):
        slots, copies = pool.append(seq, len(new_ids))
        if copies:
            src = torch.tensor([c[0] for c in copies], dtype=torch.int32, device=dev)
            dst = torch.tensor([c[1] for c in copies], dtype=torch.int32, device=dev)
            pkv.copy_blocks(kc, vc, src, dst)
        k = torch.randn(len(new_ids), Hkv, D, generator=g).to(torch.float16)
        v = torch.randn(len(new_ids), Hkv, D, generator=g).to(torch.float16)
        pkv.kv_cache_write(k.to(dev), v.to(dev), torch.tensor(slots, dtype=torch.int32, device=dev), kc, vc)
        tokens[seq] = tokens.get(seq, []) + list(new_ids)
        kk, vv = kv_tok.get(seq, (k[:0], v[:0]))
        kv_tok[seq] = (torch.cat([kk, k]), torch.cat([vv, v]))
        return copies

    prompt = list(range(1000, 1037))                      # 37 tokens: 2 full blocks + 5
    pool.add(1)
    write(1, prompt)
    pool.fork(1, 2)                                        # sequence 2 shares all three blocks
    tokens[2], kv_tok[2] = list(tokens[1]), kv_tok[1]
    assert write(1, [7, 8, 9]) != []                       # 1's shared last block is copied first
    assert write(2, [4, 5, 6, 7, 8]) == []                 # 2 now owns that block alone
    assert pool.prefix_insert(1, tokens[1]) == 2           # the two full blocks of the prompt
    assert pool.add_cached(3, prompt + [1, 2]) == 32       # 3 starts from them
    tokens[3] = prompt[:32]
    kv_tok[3] = (kv_tok[1][0][:32], kv_tok[1][1][:32])
    write(3, prompt[32:] + [1, 2, 3, 4, 5, 6])
    seqs = [1, 2, 3]
    assert pool.block_table(3)[:2] == pool.block_table(1)[:2]

    S = len(seqs)
    max_blocks = max(len(pool.block_table(s)) for s in seqs)
    bt = torch.zeros(S, max_blocks, dtype=torch.int32)
    for i, s in enumerate(seqs):
        row = pool.block_table(s)
        bt[i, :len(row)] = torch.tensor(row, dtype=torch.int32)
    ctx = torch.tensor([pool.length(s) for s in seqs], dtype=torch.int32)
    q = torch.randn(S * n, Hq, D, generator=g).to(torch.float16)
    out = torch.full_like(q, float("nan")).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_attention_decode(out, q.to(dev), kc, vc, bt.to(dev), ctx.to(dev), n, scale, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().double()
    for i, s in enumerate(seqs):
        k, v = kv_tok[s]
        assert k.shape[0] == int(ctx[i])
        if kv == "e5m2":
            k, v = k.to(torch.float8_e5m2).to(torch.float16), v.to(torch.float8_e5m2).to(torch.float16)
        ref = _dense_attention(q[i * n:(i + 1) * n], k, v, scale, n)
        import _gpu
        _gpu.compare(out[i * n:(i + 1) * n], ref.numpy(), label=f"block pool {kv} seq {s}")
    pool.close()
