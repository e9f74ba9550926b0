"""Expert cache on the GPU: a pinned-host expert bank streamed into a device slot pool.

The slot choice of every prefetch / acquire must equal the CPU LRU simulator's
exactly (same hits, misses and slots), the resident slot bytes must equal the bank
bytes, and a layer computed from the cache slots (a per-expert pointer table) must
give the same bits as the same layer computed from contiguous weights.
"""
import numpy as np
import pytest

import oracle
from synth import make_layer, stream_trace
from tests._util import bf16_tensor, ensure_built

pytestmark = pytest.mark.gpu

LAYERS, E, K, H, I, SLOTS = 3, 8, 2, 256, 128, 3


@pytest.fixture(scope="module")
def env(cuda_device):
    ensure_built()
    import torch
    from quantized_expert_ffn_layer_b300 import ftmoe as F
    return F, torch, cuda_device


def _bank(env, qtype):
    """Per layer: the layer inputs, its device weights (MoELayer) and its expert blobs."""
    F, torch, dev = env
    from quantized_expert_ffn_layer_b300 import MoELayer
    layers = []
    for l in range(LAYERS):
        L = make_layer(H=H, I=I, E=E, k=K, T=1, qtype=qtype, seed=100 + l)
        m = MoELayer(qtype, E, H, I, L.w13, L.w2, device=dev)
        blobs = torch.cat([m.w13.view(E, -1), m.w2.view(E, -1)], dim=1).contiguous()
        layers.append((L, m, blobs))
    nb = layers[0][2].shape[1]
    assert nb == F.ftmoe_expert_blob_bytes(qtype, H, I)
    bank = torch.empty((LAYERS, E, nb), dtype=torch.uint8).pin_memory()
    for l, (_, _, blobs) in enumerate(layers):
        bank[l].copy_(blobs.cpu())
    return layers, bank, nb


@pytest.mark.parametrize("policy", ["layer", "global"])
def test_cache_matches_lru_simulator_and_contiguous_layer(env, policy):
    F, torch, dev = env
    layers, bank, nb = _bank(env, "q4_0")
    pool = torch.zeros(LAYERS * SLOTS * nb, dtype=torch.uint8, device=dev)
    copy_stream = torch.cuda.Stream(dev)
    compute = torch.cuda.current_stream(dev)
    pol = F.LRU_PER_LAYER if policy == "layer" else F.LRU_GLOBAL
    cache = F.ExpertCache(LAYERS, E, nb, bank, pool, SLOTS, pol, copy_stream)
    sim = oracle.LRUSim(LAYERS, E, SLOTS, policy)
    steps = 12
    trace = stream_trace(7, steps, LAYERS, E, K, p_repeat=0.5, s=1.0)
    misses = hits = 0
    for st in range(steps):
        # prefetch layer 0 of the step, then per layer: prefetch the next, acquire this one
        pslots, pcopied = cache.prefetch(0, trace[st, 0])
        want = sim.prefetch(0, trace[st, 0])
        assert [s for s, _ in want] == pslots and [c for _, c in want] == pcopied
        for l in range(LAYERS):
            if l + 1 < LAYERS:
                pslots, pcopied = cache.prefetch(l + 1, trace[st, l + 1])
                want = sim.prefetch(l + 1, trace[st, l + 1])
                assert [s for s, _ in want] == pslots and [c for _, c in want] == pcopied
            blob_ptrs, slots, copied = cache.acquire(l, trace[st, l], compute)
            want = sim.acquire(l, trace[st, l])
            assert [s for s, _ in want] == slots and [c for _, c in want] == copied
            misses += sum(copied)
            hits += len(copied) - sum(copied)
            # the layer on one token whose routing picks exactly the acquired experts
            L, m, _ = layers[l]
            logits = np.full((1, E), -4.0, dtype=np.float32)
            logits[0, trace[st, l, 0]] = 2.0
            logits[0, trace[st, l, 1]] = 1.0
            lg = torch.from_numpy(logits).to(dev)
            x = bf16_tensor(L.x, dev)
            table = [blob_ptrs[e] if e in set(int(v) for v in trace[st, l]) else None for e in range(E)]
            wt = F.make_weights("q4_0", E, H, I, expert_blob=table)
            ws = m.workspace(1, K)
            out = torch.empty((1, H), dtype=torch.bfloat16, device=dev)
            F.ftmoe_layer(wt, lg, x, 1, K, out, None, None, ws, ws.numel())
            cache.release(l, compute)
            sim.release(l)
            ref = m.forward(lg, x, K)
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), (st, l)
    stats = cache.stats()
    assert stats["misses"] == misses and stats["hits"] == hits
    assert stats["lookups"] == steps * LAYERS * K
    assert stats["h2d_bytes"] == nb * (stats["misses"] + stats["prefetch_copies"])
    # every resident slot holds exactly its expert's bank bytes
    torch.cuda.synchronize()
    pool_h = pool.view(-1, nb).cpu()
    nslot = SLOTS if policy == "layer" else SLOTS * LAYERS
    for (l, e), s in sim.where.items():
        gs = (l * nslot + s) if policy == "layer" else s
        assert torch.equal(pool_h[gs], bank[l, e]), (l, e, s)
    cache.close()


def test_cache_rejects_requests_larger_than_the_pool(env):
    F, torch, dev = env
    layers, bank, nb = _bank(env, "mxfp4")
    pool = torch.zeros(LAYERS * SLOTS * nb, dtype=torch.uint8, device=dev)
    cache = F.ExpertCache(LAYERS, E, nb, bank, pool, SLOTS, F.LRU_PER_LAYER, torch.cuda.Stream(dev))
    with pytest.raises(F.FtmoeError) as ei:
        cache.prefetch(0, [0, 1, 2, 3])  # 4 ids, 3 slots
    assert ei.value.status == 4  # FTMOE_ERR_NO_SLOT
    with pytest.raises(F.FtmoeError) as ei:
        cache.prefetch(0, [0, E])  # expert id out of range
    assert ei.value.status == 1
    cache.close()


@pytest.mark.parametrize("policy", ["layer", "global"])
def test_history_prefetch_matches_simulator(env, policy):
    """Predictive prefetch from routing history: at each layer, prefetch what the next
    layer asked for at its previous acquire, then acquire this layer's true ids.  Every
    slot choice, hit and miss must equal the LRU simulator driven by the same requests."""
    F, torch, dev = env
    layers, bank, nb = _bank(env, "q4_0")
    pool = torch.zeros(LAYERS * SLOTS * nb, dtype=torch.uint8, device=dev)
    pol = F.LRU_PER_LAYER if policy == "layer" else F.LRU_GLOBAL
    cache = F.ExpertCache(LAYERS, E, nb, bank, pool, SLOTS, pol, torch.cuda.Stream(dev))
    sim = oracle.LRUSim(LAYERS, E, SLOTS, policy)
    compute = torch.cuda.current_stream(dev)
    steps = 10
    trace = stream_trace(9, steps, LAYERS, E, K, p_repeat=0.6, s=1.0)
    last = {}
    for st in range(steps):
        for l in range(LAYERS):
            nxt = (l + 1) % LAYERS
            ids, slots, copied = cache.prefetch_history(nxt)
            assert ids == last.get(nxt, [])
            if ids:
                want = sim.prefetch(nxt, ids)
                assert [s for s, _ in want] == slots and [c for _, c in want] == copied
            _, slots, copied = cache.acquire(l, trace[st, l], compute)
            want = sim.acquire(l, trace[st, l])
            assert [s for s, _ in want] == slots and [c for _, c in want] == copied
            last[l] = [int(v) for v in trace[st, l]]
            cache.release(l, compute)
            sim.release(l)
    torch.cuda.synchronize()
    pool_h = pool.view(-1, nb).cpu()
    nslot = SLOTS if policy == "layer" else SLOTS * LAYERS
    for (l, e), s in sim.where.items():
        gs = (l * nslot + s) if policy == "layer" else s
        assert torch.equal(pool_h[gs], bank[l, e]), (l, e, s)
    cache.close()


def test_acquired_slots_are_not_overwritten_before_release(env):
    """A global pool of E + 2 slots (less than two layers of experts): layer 0 acquires
    all E experts and, before it runs, layer 1's prefetch of all E is refused with
    NO_SLOT instead of overwriting slots layer 0 is about to read; a prefetch that fits
    the two unpinned slots succeeds.  Layer 0 computed from its slots equals the layer
    from contiguous weights bit for bit; after the release, layer 1 is fetched, acquired
    and checked the same way.  Every slot choice equals the simulator's."""
    F, torch, dev = env
    layers, bank, nb = _bank(env, "q4_0")
    nl = 2
    pool = torch.zeros((E + 2) * nb, dtype=torch.uint8, device=dev)
    copy_stream = torch.cuda.Stream(dev)
    compute = torch.cuda.current_stream(dev)
    # slots_per_layer * layers = E + 2 slots in the one global pool
    cache = F.ExpertCache(nl, E, nb, bank, pool, (E + 2) // nl,
                          F.LRU_GLOBAL, copy_stream)
    sim = oracle.LRUSim(nl, E, (E + 2) // nl, "global")
    everyone = list(range(E))

    def run_from_slots(l, blob_ptrs):
        L, m, _ = layers[l]
        lg = torch.from_numpy(np.random.default_rng(l).standard_normal((16, E)).astype(np.float32)).to(dev)
        x = bf16_tensor(np.repeat(L.x, 16, axis=0), dev)
        wt = F.make_weights("q4_0", E, H, I, expert_blob=blob_ptrs)
        ws = m.workspace(16, K)
        out = torch.empty((16, H), dtype=torch.bfloat16, device=dev)
        F.ftmoe_layer(wt, lg, x, 16, K, out, None, None, ws, ws.numel())
        return out, m.forward(lg, x, K)

    blobs, slots, copied = cache.acquire(0, everyone, compute)
    assert [(s, c) for s, c in zip(slots, copied)] == sim.acquire(0, everyone)
    with pytest.raises(F.FtmoeError) as ei:
        cache.prefetch(1, everyone)
    assert ei.value.status == 4  # FTMOE_ERR_NO_SLOT
    with pytest.raises(oracle.cache.NoSlot):
        sim.prefetch(1, everyone)
    pslots, pcopied = cache.prefetch(1, [3, 5])
    assert list(zip(pslots, pcopied)) == sim.prefetch(1, [3, 5])
    out, ref = run_from_slots(0, blobs)
    cache.release(0, compute)
    sim.release(0)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    pslots, pcopied = cache.prefetch(1, everyone)
    assert list(zip(pslots, pcopied)) == sim.prefetch(1, everyone)
    blobs, slots, copied = cache.acquire(1, everyone, compute)
    assert list(zip(slots, copied)) == sim.acquire(1, everyone)
    out, ref = run_from_slots(1, blobs)
    cache.release(1, compute)
    sim.release(1)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    st = cache.stats()
    assert st["h2d_bytes"] == nb * (st["misses"] + st["prefetch_copies"])
    cache.close()


def test_stream_workload_trace_matches_simulator(env):
    """The stream workload's bookkeeping at its full size: 48 layers of 128 experts, 32
    slots per layer, the 2048-step batch-1 trace (ids repeat with p = 0.7, else Zipf 1.0),
    the next layer prefetched while this one is acquired and released.  Every slot, hit
    and miss of the library equals the simulator's; the totals match, and every resident
    slot holds its blob's bytes (small stand-in blobs: the bytes' path is what is checked)."""
    F, torch, dev = env
    from synth import CONFIGS
    c = CONFIGS["stream"]
    layers, E, k, slots, steps = c["layers"], c["E"], c["k"], c["slots"], c["steps"]
    nb = 256
    rng = np.random.default_rng(5)
    bank = torch.from_numpy(rng.integers(0, 256, size=(layers, E, nb), dtype=np.uint8)).pin_memory()
    pool = torch.zeros(layers * slots * nb, dtype=torch.uint8, device=dev)
    cache = F.ExpertCache(layers, E, nb, bank, pool, slots, F.LRU_PER_LAYER, torch.cuda.Stream(dev))
    sim = oracle.LRUSim(layers, E, slots, "layer")
    compute = torch.cuda.current_stream(dev)
    trace = stream_trace(c["seed"], steps, layers, E, k, c["p_repeat"], c["zipf"]).tolist()
    copies = 0
    for st in range(steps):
        got = [cache.prefetch(0, trace[st][0])[:2]]
        want = [sim.prefetch(0, trace[st][0])]
        for l in range(layers):
            if l + 1 < layers:
                got.append(cache.prefetch(l + 1, trace[st][l + 1]))
                want.append(sim.prefetch(l + 1, trace[st][l + 1]))
            got.append(cache.acquire(l, trace[st][l], compute)[1:])
            want.append(sim.acquire(l, trace[st][l]))
            cache.release(l, compute)
            sim.release(l)
        for (gs, gc), w in zip(got, want):
            assert list(zip(gs, gc)) == w, st
            copies += sum(gc)
    stats = cache.stats()
    assert stats["lookups"] == steps * layers * k
    assert stats["misses"] + stats["prefetch_copies"] == copies
    assert stats["h2d_bytes"] == nb * copies
    torch.cuda.synchronize()
    pool_h = pool.view(-1, nb).cpu()
    for (l, e), s in sim.where.items():
        assert torch.equal(pool_h[l * slots + s], bank[l, e]), (l, e, s)
    cache.close()
