"""LRU expert-slot cache simulator (host bookkeeping only, no data).

[P3] 机制四 and [P5] §五: hot experts stay resident in GPU memory, cold ones live
in pinned host memory, and an LRU decides which resident expert to evict;
[P3] 机制一 / [P4] 方法: the next layer's weights are copied while the current
layer computes.  The pages do not define the bookkeeping; the readings are:

* a pool of slots per layer ("layer" policy) or one pool for all layers
  ("global" policy, the pages' "global LRU");
* every request (a prefetch or an acquire of a list of expert ids for a layer)
  touches its ids in order; each touch takes the next value of one global use
  counter as the slot's recency stamp;
* a touched expert that is resident is a hit; otherwise it is copied into the
  lowest-numbered empty slot of its pool, else into the slot with the smallest
  stamp, never into a slot already touched by the same request and never into a
  pinned slot (no such slot left -> "no slot");
* an acquire (the request a layer makes right before it runs) pins the slots it
  touched until that layer's release, so that a later prefetch or acquire cannot
  overwrite weights the layer is about to read or is reading ([P4] 核心洞察: the LRU
  serves a layer replayed as a CUDA graph, which reads its experts' slots in place);
  a prefetch pins nothing;
* a request that fails with "no slot" changes nothing (it is all or nothing).
"""
from __future__ import annotations


class NoSlot(RuntimeError):
    pass


class LRUSim:
    def __init__(self, layers: int, E: int, slots_per_layer: int, policy: str = "layer"):
        if policy not in ("layer", "global"):
            raise ValueError(policy)
        self.layers, self.E, self.policy = layers, E, policy
        self.npools = layers if policy == "layer" else 1
        self.nslot = slots_per_layer if policy == "layer" else slots_per_layer * layers
        self.owner = [[None] * self.nslot for _ in range(self.npools)]
        self.stamp = [[0] * self.nslot for _ in range(self.npools)]
        self.pins = [[0] * self.nslot for _ in range(self.npools)]
        self.pinned_by: dict[int, list[int]] = {}  # layer -> slots its acquires pinned
        self.where: dict[tuple[int, int], int] = {}
        self.clock = 0

    def pool_of(self, layer: int) -> int:
        return layer if self.policy == "layer" else 0

    def request(self, layer: int, ids, pin: bool = False) -> list[tuple[int, bool]]:
        """Touch ``ids`` of ``layer``; returns [(slot, copied)] per id (slot is the index
        inside the layer's pool, or inside the single pool for the global policy).  With
        ``pin`` the touched slots stay pinned until ``release(layer)``.  Raises NoSlot,
        leaving every record as it was, when a missing id finds no slot to take."""
        pool = self.pool_of(layer)
        owner, stamp, pins = self.owner[pool], self.stamp[pool], self.pins[pool]
        saved = (list(owner), list(stamp), dict(self.where), self.clock)
        touched: set[int] = set()
        out = []
        for e in ids:
            e = int(e)
            key = (layer, e)
            self.clock += 1
            if key in self.where:
                s, copied = self.where[key], False
            else:
                free = [s for s in range(self.nslot) if s not in touched and pins[s] == 0]
                if not free:
                    owner[:], stamp[:] = saved[0], saved[1]
                    self.where, self.clock = saved[2], saved[3]
                    raise NoSlot(f"layer {layer}: no unpinned slot left for expert {e}")
                empty = [s for s in free if owner[s] is None]
                s = empty[0] if empty else min(free, key=lambda q: stamp[q])
                if owner[s] is not None:
                    del self.where[owner[s]]
                owner[s] = key
                self.where[key] = s
                copied = True
            stamp[s] = self.clock
            touched.add(s)
            out.append((s, copied))
        if pin:
            for s in sorted(touched):
                pins[s] += 1
                self.pinned_by.setdefault(layer, []).append(s)
        return out

    def prefetch(self, layer: int, ids) -> list[tuple[int, bool]]:
        return self.request(layer, ids, pin=False)

    def acquire(self, layer: int, ids) -> list[tuple[int, bool]]:
        return self.request(layer, ids, pin=True)

    def release(self, layer: int) -> None:
        """Unpins the slots of every acquire of ``layer`` since its previous release."""
        pins = self.pins[self.pool_of(layer)]
        for s in self.pinned_by.pop(layer, []):
            pins[s] -= 1
