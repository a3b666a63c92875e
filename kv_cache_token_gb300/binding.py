"""ctypes binding of libkvevict.so: argument marshalling only.

Every method has the name of the C entry point it calls (kvevict_<name>) and
passes raw device pointers and the current torch CUDA stream.  Device memory
for the engine state is owned by the Engine object (torch tensors sized by
kvevict_buffer_size); the library never allocates.
"""
import ctypes
import os

import torch

H2O, SNAPKV, DROPKV = 0, 1, 2
BF16, F32 = 0, 1
KEY_F32, KEY_F64 = 0, 1

STATUS = {0: "OK", 1: "E_INVALID_ARG", 2: "E_POOL_KERNEL_EVEN", 3: "E_RECENT_GE_BUDGET",
          4: "E_OBS_WINDOW_ZERO", 5: "E_NO_BLOCKS", 6: "E_DTYPE", 7: "E_CUDA", 8: "E_TIMEOUT",
          9: "E_DEVICE", 10: "E_SCRATCH_LIMIT"}
STAT_NAMES = ["steps", "victims", "admit_new_block", "freed_dead", "freed_reloc", "moved", "plans",
              "deferred", "nan_keys", "blocks", "live", "half_empty", "lanes"]
NSTATS = len(STAT_NAMES)
(BUF_K_POOL, BUF_V_POOL, BUF_POSITIONS, BUF_SLOTS, BUF_COUNTS, BUF_SCORES, BUF_RING, BUF_RING_SLOT,
 BUF_BLOCK_OWNER, BUF_BLOCK_MASK, BUF_LANE_BLOCKS, BUF_LANE_NBLOCKS, BUF_STATS, BUF_WORKSPACE) = range(14)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvevict.so")


class KvevictError(RuntimeError):
    def __init__(self, code, what):
        super().__init__("%s: %s" % (what, STATUS.get(code, code)))
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "policy", "num_layers", "batch", "num_q_heads", "num_kv_heads", "head_dim", "kv_dtype",
        "block_size", "blocks_per_pool", "max_tokens", "budget", "recent_window", "obs_window",
        "pool_kernel")] + [("theta_f", ctypes.c_float), ("max_window", ctypes.c_int32)]


class Buffers(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "k_pool", "v_pool", "positions", "slots", "counts", "scores", "ring", "ring_slot",
        "block_owner", "block_mask", "lane_blocks", "lane_nblocks", "stats", "workspace")]


_LIB = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libkvevict.so is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, V = ctypes.POINTER, ctypes.c_int32, ctypes.c_void_p
        L.kvevict_validate.argtypes = [P(Config)]
        L.kvevict_buffer_size.argtypes = [P(Config), ctypes.c_int]
        L.kvevict_buffer_size.restype = ctypes.c_size_t
        L.kvevict_workspace_size.argtypes = [P(Config)]
        L.kvevict_workspace_size.restype = ctypes.c_size_t
        L.kvevict_create.argtypes = [P(Config), P(Buffers), P(V)]
        L.kvevict_destroy.argtypes = [V]
        L.kvevict_destroy.restype = None
        L.kvevict_reset.argtypes = [V, V]
        L.kvevict_set_layer_budget.argtypes = [V, ctypes.c_int, I, I]
        L.kvevict_prefill.argtypes = [V, ctypes.c_int, V, V, I, V]
        L.kvevict_decode_step.argtypes = [V, ctypes.c_int, V, V, V, I, V, V, V, V, V]
        L.kvevict_attend.argtypes = [V, ctypes.c_int, V, V, V, V]
        L.kvevict_finish_step.argtypes = [V, ctypes.c_int, V, V, V, I, V, V, V, V, V]
        L.kvevict_score.argtypes = [V, ctypes.c_int, V, I, V, V, V, V, V]
        L.kvevict_score_mass.argtypes = [V, ctypes.c_int, V, I, V, I, V, V, V]
        L.kvevict_attend_static.argtypes = [V, ctypes.c_int, V, V, V, V, V, V]
        L.kvevict_select.argtypes = [V, V, I, V, V, I, I, I, I, V, V, V]
        L.kvevict_compact.argtypes = [V, ctypes.c_int, V, V, V, V, V, V, V]
        L.kvevict_defer_relocation.argtypes = [V, I]
        L.kvevict_relocate.argtypes = [V, ctypes.c_int, V, V, V, V, V]
        L.kvevict_stats.argtypes = [V, ctypes.c_int, V, V]
        L.kvevict_last_error.argtypes = [V, ctypes.c_char_p, ctypes.c_size_t]
        L.kvevict_check_wait_timeout.argtypes = [V, I, V]
        L.kvevict_kernels_per_decode_step.argtypes = [V]
        L.kvevict_kernels_per_decode_step.restype = I
        for f in ("validate", "create", "reset", "set_layer_budget", "prefill", "decode_step", "attend", "finish_step",
                  "attend_static",
                  "score", "score_mass", "select",
                  "compact", "defer_relocation", "relocate", "stats", "check_wait_timeout", "last_error"):
            getattr(L, "kvevict_" + f).restype = ctypes.c_int
        _LIB = L
    return _LIB


def config_from(shape=None, **kw):
    """A Config from a workloads Shape (or keyword fields)."""
    f = {}
    if shape is not None:
        f = dict(policy=shape.policy, num_layers=shape.num_layers, batch=shape.batch,
                 num_q_heads=shape.num_q_heads, num_kv_heads=shape.num_kv_heads,
                 head_dim=shape.head_dim, kv_dtype=BF16 if shape.kv_dtype == "bf16" else F32,
                 block_size=16, blocks_per_pool=shape.blocks_per_pool,
                 max_tokens=shape.max_tokens, budget=shape.budget,
                 recent_window=shape.recent_window, obs_window=shape.obs_window,
                 pool_kernel=shape.pool_kernel, theta_f=shape.theta_f, max_window=shape.window)
    f.update(kw)
    f.setdefault("block_size", 16)
    f.setdefault("theta_f", 0.25)
    f.setdefault("max_window", 0)
    return Config(**f)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(code, what):
    if code != 0:
        raise KvevictError(code, what)


def validate(cfg):
    return lib().kvevict_validate(ctypes.byref(cfg))


class Engine:
    """Device state of one engine plus the C-ABI calls on it."""

    def __init__(self, cfg, device="cuda"):
        L = lib()
        self.cfg = cfg
        _check(L.kvevict_validate(ctypes.byref(cfg)), "kvevict_validate")
        self.device = torch.device(device)
        c = cfg
        lanes = c.batch * c.num_kv_heads
        self.lanes = lanes
        self.g = c.num_q_heads // c.num_kv_heads
        kvdt = torch.bfloat16 if c.kv_dtype == BF16 else torch.float32
        self.kv_dtype = kvdt
        dev = self.device

        def buf(which, shape, dtype):
            nbytes = L.kvevict_buffer_size(ctypes.byref(cfg), which)
            t = torch.empty(shape, dtype=dtype, device=dev)
            assert t.numel() * t.element_size() == nbytes, (which, nbytes, t.numel() * t.element_size())
            return t

        Lr, P, C, d = c.num_layers, c.blocks_per_pool, c.max_tokens, c.head_dim
        self.k_pool = buf(BUF_K_POOL, (Lr, P, 16, d), kvdt)
        self.v_pool = buf(BUF_V_POOL, (Lr, P, 16, d), kvdt)
        self.positions = buf(BUF_POSITIONS, (Lr, lanes, C), torch.int32)
        self.slots = buf(BUF_SLOTS, (Lr, lanes, C), torch.int32)
        self.counts = buf(BUF_COUNTS, (Lr, lanes), torch.int32)
        self.scores = buf(BUF_SCORES, (Lr, lanes, C), torch.float32)
        # history rows sit at the tokens' slots: ring[layer][slot] (slot = block * 16 + offset)
        self.ring = (buf(BUF_RING, (Lr, P * 16, c.obs_window), torch.float32)
                     if c.policy == SNAPKV or (c.policy == DROPKV and c.obs_window >= 1) else None)
        self.ring_slot = buf(BUF_RING_SLOT, (Lr, lanes), torch.int32)
        self.block_owner = buf(BUF_BLOCK_OWNER, (Lr, P), torch.int32)
        self.block_mask = buf(BUF_BLOCK_MASK, (Lr, P), torch.int32)
        self.lane_blocks = buf(BUF_LANE_BLOCKS, (Lr, lanes, C), torch.int32)
        self.lane_nblocks = buf(BUF_LANE_NBLOCKS, (Lr, lanes), torch.int32)
        self.stats_buf = buf(BUF_STATS, (Lr, NSTATS), torch.int64)
        ws = L.kvevict_workspace_size(ctypes.byref(cfg))
        self.workspace = torch.empty(ws + 256, dtype=torch.uint8, device=dev)
        off = (-self.workspace.data_ptr()) % 256
        self.workspace_aligned = self.workspace[off:off + ws]
        b = Buffers(*[_ptr(t) for t in (
            self.k_pool, self.v_pool, self.positions, self.slots, self.counts, self.scores,
            self.ring, self.ring_slot, self.block_owner, self.block_mask, self.lane_blocks,
            self.lane_nblocks, self.stats_buf, self.workspace_aligned)])
        self._bufs = b
        h = ctypes.c_void_p()
        with torch.cuda.device(dev):
            _check(L.kvevict_create(ctypes.byref(cfg), ctypes.byref(b), ctypes.byref(h)), "kvevict_create")
        self.h = h
        # per-call outputs reused by default
        self.victims = torch.zeros((lanes, C), dtype=torch.int32, device=dev)
        self.n_victims = torch.zeros((lanes,), dtype=torch.int32, device=dev)

    def __del__(self):
        h = getattr(self, "h", None)
        if h is not None and _LIB is not None:
            _LIB.kvevict_destroy(h)
            self.h = None

    # ---- C-ABI calls ----------------------------------------------------------
    def reset(self, stream=None):
        _check(lib().kvevict_reset(self.h, _stream(stream)), "kvevict_reset")

    def set_layer_budget(self, layer, budget, recent_window):
        """kvevict_set_layer_budget: later decode steps of `layer` keep `budget` tokens."""
        _check(lib().kvevict_set_layer_budget(self.h, layer, budget, recent_window), "kvevict_set_layer_budget")

    def prefill(self, layer, k_ctx, v_ctx, stream=None):
        assert k_ctx.is_contiguous() and v_ctx.is_contiguous() and k_ctx.dtype == self.kv_dtype
        n = k_ctx.shape[2]
        _check(lib().kvevict_prefill(self.h, layer, _ptr(k_ctx), _ptr(v_ctx), n, _stream(stream)),
               "kvevict_prefill")

    def decode_step(self, layer, q, k_new, v_new, new_pos, out=None, lse=None, victims=None,
                    n_victims=None, stream=None):
        c = self.cfg
        if q is not None and out is None:
            out = torch.empty((c.batch, c.num_q_heads, c.head_dim), dtype=torch.float32, device=self.device)
        if q is not None and lse is None:
            lse = torch.empty((c.batch, c.num_q_heads), dtype=torch.float32, device=self.device)
        victims = self.victims if victims is None else victims
        n_victims = self.n_victims if n_victims is None else n_victims
        for t in (q, k_new, v_new):
            assert t is None or (t.is_contiguous() and t.dtype == self.kv_dtype)
        _check(lib().kvevict_decode_step(self.h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), int(new_pos),
                                         _ptr(out), _ptr(lse), _ptr(victims), _ptr(n_victims),
                                         _stream(stream)), "kvevict_decode_step")
        return out, lse, victims, n_victims

    def attend(self, layer, q, k_new, v_new, stream=None):
        _check(lib().kvevict_attend(self.h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _stream(stream)),
               "kvevict_attend")

    def finish_step(self, layer, q, k_new, v_new, new_pos, out=None, lse=None, victims=None, n_victims=None,
                    stream=None):
        c = self.cfg
        if q is not None and out is None:
            out = torch.empty((c.batch, c.num_q_heads, c.head_dim), dtype=torch.float32, device=self.device)
        if q is not None and lse is None:
            lse = torch.empty((c.batch, c.num_q_heads), dtype=torch.float32, device=self.device)
        victims = self.victims if victims is None else victims
        n_victims = self.n_victims if n_victims is None else n_victims
        _check(lib().kvevict_finish_step(self.h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), int(new_pos),
                                         _ptr(out), _ptr(lse), _ptr(victims), _ptr(n_victims),
                                         _stream(stream)), "kvevict_finish_step")
        return out, lse, victims, n_victims

    def attend_static(self, layer, q, k_new, v_new, out=None, lse=None, stream=None):
        """kvevict_attend_static: attention output and LSE of one layer using the
        library's built-in scratch array (no workspace, no allocation inside)."""
        c = self.cfg
        if out is None:
            out = torch.empty((c.batch, c.num_q_heads, c.head_dim), dtype=torch.float32, device=self.device)
        if lse is None:
            lse = torch.empty((c.batch, c.num_q_heads), dtype=torch.float32, device=self.device)
        _check(lib().kvevict_attend_static(self.h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out), _ptr(lse),
                                           _stream(stream)), "kvevict_attend_static")
        return out, lse

    def score(self, layer, q_win, q_pos, lse=None, a_out=None, scores=None, stream=None):
        c = self.cfg
        if q_win is None:
            _check(lib().kvevict_score(self.h, layer, None, 0, None, None, None, None, _stream(stream)),
                   "kvevict_score")
            return None
        w = q_win.shape[2]
        if lse is None:
            lse = torch.empty((c.batch, c.num_q_heads, w), dtype=torch.float32, device=self.device)
        if a_out is None:
            a_out = torch.empty((c.batch, c.num_q_heads, w, c.head_dim), dtype=torch.float32, device=self.device)
        if scores is None:
            scores = torch.zeros((self.lanes, c.max_tokens), dtype=torch.float32, device=self.device)
        assert q_win.is_contiguous() and q_pos.dtype == torch.int32
        _check(lib().kvevict_score(self.h, layer, _ptr(q_win), w, _ptr(q_pos), _ptr(lse), _ptr(a_out),
                                   _ptr(scores), _stream(stream)), "kvevict_score")
        return lse, a_out, scores

    def score_mass(self, layer, q_win, q_pos, kind, lse=None, scores=None, stream=None):
        """kvevict_score_mass; kind 0 = SnapKV prefill keys, 1 = H2O
        causal-prefill scores.  Returns (lse, scores) or None for q_win None."""
        c = self.cfg
        if q_win is None:
            _check(lib().kvevict_score_mass(self.h, layer, None, 0, None, kind, None, None, _stream(stream)),
                   "kvevict_score_mass")
            return None
        w = q_win.shape[2]
        if lse is None:
            lse = torch.empty((c.batch, c.num_q_heads, w), dtype=torch.float32, device=self.device)
        if scores is None:
            scores = torch.zeros((self.lanes, c.max_tokens), dtype=torch.float32, device=self.device)
        assert q_win.is_contiguous() and q_pos.dtype == torch.int32
        _check(lib().kvevict_score_mass(self.h, layer, _ptr(q_win), w, _ptr(q_pos), kind, _ptr(lse),
                                        _ptr(scores), _stream(stream)), "kvevict_score_mass")
        return lse, scores

    def select(self, keys, positions, counts, budget, recent_window, victims=None, n_victims=None,
               stream=None):
        n_lanes, stride = keys.shape
        kd = KEY_F64 if keys.dtype == torch.float64 else KEY_F32
        if victims is None:
            victims = torch.full((n_lanes, stride), -1, dtype=torch.int32, device=self.device)
        if n_victims is None:
            n_victims = torch.zeros((n_lanes,), dtype=torch.int32, device=self.device)
        assert keys.is_contiguous() and positions.is_contiguous() and positions.shape == keys.shape
        _check(lib().kvevict_select(self.h, _ptr(keys), kd, _ptr(positions), _ptr(counts), n_lanes, stride,
                                    budget, recent_window, _ptr(victims), _ptr(n_victims), _stream(stream)),
               "kvevict_select")
        return victims, n_victims

    def compact(self, layer, victims, n_victims, freed=None, n_freed=None, moves=None, n_moves=None,
                stream=None):
        c = self.cfg
        # the library writes freed[0..n_freed) and moves[0..n_moves) and both counts
        if freed is None:
            freed = torch.empty((c.blocks_per_pool,), dtype=torch.int32, device=self.device)
        if n_freed is None:
            n_freed = torch.empty((1,), dtype=torch.int32, device=self.device)
        if moves is None:
            moves = torch.empty((self.lanes * c.max_tokens, 6), dtype=torch.int32, device=self.device)
        if n_moves is None:
            n_moves = torch.empty((1,), dtype=torch.int32, device=self.device)
        _check(lib().kvevict_compact(self.h, layer, _ptr(victims), _ptr(n_victims), _ptr(freed), _ptr(n_freed),
                                     _ptr(moves), _ptr(n_moves), _stream(stream)), "kvevict_compact")
        return freed, n_freed, moves, n_moves

    def defer_relocation(self, deferred=True):
        """kvevict_defer_relocation: decode steps plan no relocation while set."""
        _check(lib().kvevict_defer_relocation(self.h, 1 if deferred else 0), "kvevict_defer_relocation")

    def relocate(self, layer, freed=None, n_freed=None, moves=None, n_moves=None, stream=None):
        """kvevict_relocate on `stream`; returns (freed, n_freed, moves, n_moves)."""
        c = self.cfg
        if freed is None:
            freed = torch.empty((c.blocks_per_pool,), dtype=torch.int32, device=self.device)
        if n_freed is None:
            n_freed = torch.empty((1,), dtype=torch.int32, device=self.device)
        if moves is None:
            moves = torch.empty((self.lanes * c.max_tokens, 6), dtype=torch.int32, device=self.device)
        if n_moves is None:
            n_moves = torch.empty((1,), dtype=torch.int32, device=self.device)
        _check(lib().kvevict_relocate(self.h, layer, _ptr(freed), _ptr(n_freed), _ptr(moves), _ptr(n_moves),
                                      _stream(stream)), "kvevict_relocate")
        return freed, n_freed, moves, n_moves

    def stats(self, layer, stream=None):
        out = torch.zeros((NSTATS,), dtype=torch.int64, device=self.device)
        _check(lib().kvevict_stats(self.h, layer, _ptr(out), _stream(stream)), "kvevict_stats")
        return out

    def kernels_per_decode_step(self):
        """kvevict_kernels_per_decode_step (2 or 3)."""
        return int(lib().kvevict_kernels_per_decode_step(self.h))

    def check_wait_timeout(self, polls, stream=None):
        """kvevict_check_wait_timeout: the next last_error() reports a timeout."""
        _check(lib().kvevict_check_wait_timeout(self.h, polls, _stream(stream)), "kvevict_check_wait_timeout")

    def last_error(self):
        buf = ctypes.create_string_buffer(256)
        code = lib().kvevict_last_error(self.h, buf, 256)
        return code, buf.value.decode()
