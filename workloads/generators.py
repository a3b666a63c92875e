"""Seeded generators for the five synthetic workloads.

Every tensor is drawn from a torch.Generator whose seed mixes the workload
seed with a purpose tag, the layer and the step, so any piece can be
regenerated alone and on either device.  K/V/q are rounded to the workload's
storage dtype (bf16 or fp32) before anyone sees them, so the CUDA path and
the oracle read identical bits.

Workloads (shapes from the task's five configs; the constructions marked
"chosen" are readings where the configs are silent):

1. h2o_toy: B=1, Hq=Hkv=1, d=64, fp32, context 512, q/K/V ~ N(0,1); 32 decode
   steps with fresh N(0,1) q, k, v; budget 128 = 64 heavy + 64 recent.
2. snapkv_decode: B=4, Hq=32, Hkv=8, d=128, bf16, context 4096; K ~ N(0,1);
   per (b, kvh) a direction u = q*/|q*| with q* ~ N(0,I) (chosen); 40
   non-overlapping runs of U{8..32} tokens at uniform starts (redrawn on
   overlap; scaled copies plant 40 * ctx / 4096 runs) get k += 3u; decode queries q_h = q* + N(0,I) (chosen) so a run
   token's logit is lifted by about 3; V ~ N(0,1); obsWindow 32,
   poolKernel 7, recentWindow 256, budget 1024, 256 steps.
3. dropkv_prefill: B=1, Hq=32, Hkv=8, d=128, bf16, context 32768; q/K/V ~
   N(0,1) with 1% of key positions per lane (uniform draw) scaled x4; window =
   the last 64 positions; keep floor(5%) = 1638 per KV head.
4. h2o_70b: 80 layers, Hkv=8, Hq=64 (group 8: a Llama-70B-shaped assumption),
   d=128, bf16, B=16, context 16384 (~86 GB of K/V); per (layer, b, kvh) a
   unit u and a random rank permutation pi; k_j = (-1.1 ln pi_j) u + z_j -
   (z_j.u) u with z ~ N(0,I); decode q_h = sqrt(d) u + N(0, 0.1^2 I), so the
   logit of rank r is about -1.1 ln r (Zipf s = 1.1 weights); new tokens draw
   a uniform rank; V ~ N(0,1); budget floor(20%) = 3276 with recent 1638;
   64 decode steps.
5. paged_128k: as 3 with context 131072 (8192 blocks per lane), keep
   floor(5%) = 6553, then forced compaction.
6. snapkv_prefill / snapkv_prefill_128k (SnapKV's own one-shot prefill
   selection, which the SnapKV page describes; sizes chosen): B=1, Hq=32,
   Hkv=8, d=128, bf16, context 32768 / 131072; keys and planted runs as in 2
   (40 runs per 4096 tokens); the last 32 prompt positions are the
   observation window (the H2O Guide's "last 32 prompt tokens"), their
   queries q* + N(0,I) as in 2's decode queries; poolKernel 7; keep 1/16 of
   the prompt (2048 / 8192, the H2O Guide's 64,000 -> 4,000 ratio) with the
   window protected.
"""
import dataclasses
import math

import torch

H2O, SNAPKV, DROPKV = 0, 1, 2
BLOCK = 16


@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    policy: int
    num_layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str          # "bf16" | "fp32"
    ctx: int
    steps: int
    budget: int
    recent_window: int
    obs_window: int
    pool_kernel: int
    seed: int
    window: int = 0        # DropKV prefill window (query rows per head)
    theta_f: float = 0.25
    kind: str = "decode"   # "decode" | "prefill"

    @property
    def lanes(self):
        return self.batch * self.num_kv_heads

    @property
    def group(self):
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_tokens(self):
        """Token-table capacity per lane: the context plus every token a
        lane could gain before it first reaches the budget, plus the token
        being admitted."""
        return self.ctx + self.steps + 1

    @property
    def blocks_per_pool(self):
        """Blocks of one layer's pool: every lane's full table, plus headroom
        for relocation destinations (at most ceil(budget/16) + 1 per lane)."""
        per_lane = -(-self.max_tokens // BLOCK) + -(-self.budget // BLOCK) + 2
        return self.lanes * per_lane

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.kv_dtype == "bf16" else torch.float32

    @property
    def kv_bytes(self):
        """K+V bytes of the full context (2 x 2 x L x Hkv x d x ctx x B for bf16)."""
        es = 2 if self.kv_dtype == "bf16" else 4
        return 2 * es * self.num_layers * self.num_kv_heads * self.head_dim * self.ctx * self.batch


SHAPES = {
    "h2o_toy": Shape("h2o_toy", H2O, 1, 1, 1, 1, 64, "fp32", 512, 32, 128, 64, 1, 1, seed=1),
    "snapkv_decode": Shape("snapkv_decode", SNAPKV, 1, 4, 32, 8, 128, "bf16", 4096, 256,
                           1024, 256, 32, 7, seed=2),
    "dropkv_prefill": Shape("dropkv_prefill", DROPKV, 1, 1, 32, 8, 128, "bf16", 32768, 0,
                            1638, 64, 1, 1, seed=3, window=64, kind="prefill"),
    "h2o_70b": Shape("h2o_70b", H2O, 80, 16, 64, 8, 128, "bf16", 16384, 64,
                     3276, 1638, 1, 1, seed=4),
    "paged_128k": Shape("paged_128k", DROPKV, 1, 1, 32, 8, 128, "bf16", 131072, 0,
                        6553, 64, 1, 1, seed=5, window=64, kind="prefill"),
    "snapkv_prefill": Shape("snapkv_prefill", SNAPKV, 1, 1, 32, 8, 128, "bf16", 32768, 0,
                            2048, 32, 32, 7, seed=6, window=32, kind="prefill"),
    "snapkv_prefill_128k": Shape("snapkv_prefill_128k", SNAPKV, 1, 1, 32, 8, 128, "bf16", 131072, 0,
                                 8192, 32, 32, 7, seed=7, window=32, kind="prefill"),
}


def shape(name):
    return SHAPES[name]


def scaled(name, **changes):
    """A smaller copy of a workload (same generator, fewer layers/steps,
    shorter context, ...) for parity tests the oracle finishes in seconds.
    Budgets given as fractions keep their floor() reading."""
    base = SHAPES[name]
    return dataclasses.replace(base, name=base.name + "_scaled", **changes)


def _mix(*vals):
    """A 63-bit seed from integers (splitmix64-style finaliser)."""
    x = 0x9E3779B97F4A7C15
    for v in vals:
        x = (x ^ (int(v) & 0xFFFFFFFFFFFFFFFF)) * 0xBF58476D1CE4E5B9 & 0xFFFFFFFFFFFFFFFF
        x = (x ^ (x >> 31)) * 0x94D049BB133111EB & 0xFFFFFFFFFFFFFFFF
        x ^= x >> 29
    return x & 0x7FFFFFFFFFFFFFFF


_TAGS = {"ctx_k": 1, "ctx_v": 2, "dir": 3, "perm": 4, "runs": 5, "step_q": 6,
         "step_k": 7, "step_v": 8, "win_q": 9, "heavy": 10, "rank": 11}


class Workload:
    """Seeded inputs of one Shape."""

    def __init__(self, shp):
        self.s = shp

    def _gen(self, tag, layer=0, step=0, device="cpu"):
        g = torch.Generator(device=device)
        g.manual_seed(_mix(self.s.seed, _TAGS[tag], layer, step))
        return g

    def _randn(self, shp, tag, layer=0, step=0, device="cpu"):
        return torch.randn(shp, generator=self._gen(tag, layer, step, device), device=device,
                           dtype=torch.float32)

    def _store(self, x):
        return x.to(self.s.torch_dtype)

    # ---- per-lane structure ---------------------------------------------
    def _direction(self, layer, device):
        """Unit direction per (b, kvh) [B, Hkv, d] and the raw q* it came from."""
        s = self.s
        qstar = self._randn((s.batch, s.num_kv_heads, s.head_dim), "dir", layer, 0, device)
        u = qstar / qstar.norm(dim=-1, keepdim=True)
        return u, qstar

    def _runs(self, layer):
        """Non-overlapping planted runs per (b, kvh): 40 at context 4096,
        scaled with the context for shorter prompts; list of (start, length)."""
        s = self.s
        n_runs = max(1, round(40 * s.ctx / 4096))
        g = self._gen("runs", layer)
        out = []
        for _ in range(s.lanes):
            taken = torch.zeros(s.ctx, dtype=torch.bool)
            runs = []
            tries = 0
            while len(runs) < n_runs and tries < 100000:
                tries += 1
                ln = int(torch.randint(8, 33, (1,), generator=g))
                st = int(torch.randint(0, s.ctx - ln + 1, (1,), generator=g))
                if taken[st:st + ln].any():
                    continue
                taken[st:st + ln] = True
                runs.append((st, ln))
            out.append(runs)
        return out

    # ---- context ---------------------------------------------------------
    def context(self, layer=0, device="cpu"):
        """(K, V) of the prompt, [B, Hkv, ctx, d] in the storage dtype."""
        s = self.s
        shp = (s.batch, s.num_kv_heads, s.ctx, s.head_dim)
        V = self._randn(shp, "ctx_v", layer, 0, device)
        if s.name.startswith("h2o_70b"):
            u, _ = self._direction(layer, device)
            z = self._randn(shp, "ctx_k", layer, 0, device)
            pr = torch.rand(shp[:3], generator=self._gen("perm", layer, 0, device), device=device)
            rank = pr.argsort(dim=-1).to(torch.float32) + 1.0      # a random permutation of 1..ctx
            uu = u[:, :, None, :]
            z = z - (z * uu).sum(-1, keepdim=True) * uu
            K = (-1.1 * torch.log(rank))[..., None] * uu + z
            del z, pr, rank
        else:
            K = self._randn(shp, "ctx_k", layer, 0, device)
            if s.name.startswith("snapkv"):
                u, _ = self._direction(layer, device)
                runs = self._runs(layer)
                for lane, rl in enumerate(runs):
                    b, h = divmod(lane, s.num_kv_heads)
                    for st, ln in rl:
                        K[b, h, st:st + ln] += 3.0 * u[b, h]
            elif s.policy == DROPKV:
                n_heavy = max(1, s.ctx // 100)
                g = self._gen("heavy", layer, 0, device)
                sel = torch.rand(shp[:3], generator=g, device=device).argsort(dim=-1)[..., :n_heavy]
                scale = torch.ones(shp[:3], device=device)
                scale.scatter_(2, sel, 4.0)
                K = K * scale[..., None]
        return self._store(K), self._store(V)

    # ---- decode steps ----------------------------------------------------
    def step(self, layer, t, device="cpu"):
        """(q [B, Hq, d], k_new [B, Hkv, d], v_new [B, Hkv, d], new_pos) of
        decode step t (0-based) of ``layer``."""
        s = self.s
        d = s.head_dim
        kshape = (s.batch, s.num_kv_heads, d)
        qshape = (s.batch, s.num_q_heads, d)
        v_new = self._randn(kshape, "step_v", layer, t, device)
        if s.name.startswith("h2o_70b"):
            u, _ = self._direction(layer, device)
            ug = u.repeat_interleave(s.group, dim=1)
            q = math.sqrt(d) * ug + 0.1 * self._randn(qshape, "step_q", layer, t, device)
            z = self._randn(kshape, "step_k", layer, t, device)
            z = z - (z * u).sum(-1, keepdim=True) * u
            r = torch.randint(1, s.ctx + 1, kshape[:2], generator=self._gen("rank", layer, t, device),
                              device=device).to(torch.float32)
            k_new = (-1.1 * torch.log(r))[..., None] * u + z
        elif s.name.startswith("snapkv"):
            _, qstar = self._direction(layer, device)
            q = qstar.repeat_interleave(s.group, dim=1) + self._randn(qshape, "step_q", layer, t, device)
            k_new = self._randn(kshape, "step_k", layer, t, device)
        else:
            q = self._randn(qshape, "step_q", layer, t, device)
            k_new = self._randn(kshape, "step_k", layer, t, device)
        return self._store(q), self._store(k_new), self._store(v_new), s.ctx + t

    # ---- DropKV prefill window ---------------------------------------------
    def window(self, layer=0, device="cpu"):
        """(q_win [B, Hq, w, d], q_pos [w] int32): the last w prompt positions."""
        s = self.s
        q = self._randn((s.batch, s.num_q_heads, s.window, s.head_dim), "win_q", layer, 0, device)
        if s.name.startswith("snapkv"):
            _, qstar = self._direction(layer, device)
            q = q + qstar.repeat_interleave(s.group, dim=1)[:, :, None, :]
        pos = torch.arange(s.ctx - s.window, s.ctx, dtype=torch.int32, device=device)
        return self._store(q), pos
