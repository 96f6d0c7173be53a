"""PyTorch-facing wrapper over the C ABI, shaped like the MoonEP Python API.

"MoonEP Public API Visual Guide": Buffer(...), Buffer.dispatch(...),
Buffer.prefetch_weight(...), Buffer.combine(...), Buffer.reduce_grad(...),
the two buffer views, Buffer.destroy() and MoonEPCommPlan.clone().

The R expert-parallel ranks live on one GPU, so every tensor carries a
leading rank axis: hidden_sh is [R, S, H], topk [R, S, K], and dispatched rows
are [R*NvS, H] (rank j's window starts at row j*NvS).  Everything is issued on
torch's current CUDA stream; PyTorch provides memory and streams only, and
every step runs in libmoonep's kernels.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import MoonepCommPlan, MoonepConfig, check


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


class _DeviceArray:
    """Zero-copy, non-owning view of library-owned device memory."""

    def __init__(self, ptr: int, shape, typestr: str, owner):
        self._owner = owner
        self.__cuda_array_interface__ = {
            "shape": tuple(int(s) for s in shape), "typestr": typestr,
            "data": (int(ptr), False), "version": 3, "strides": None, "stream": None}


def _view(ptr, shape, owner, dtype=torch.int32):
    typestr = {torch.int32: "<i4", torch.float32: "<f4", torch.bfloat16: "<u2"}[dtype]
    n = 1
    for s in shape:
        n *= int(s)
    if not ptr or n == 0:
        return torch.empty(shape, dtype=dtype, device="cuda")
    t = torch.as_tensor(_DeviceArray(ptr, shape, typestr, owner), device="cuda")
    if dtype == torch.bfloat16:
        t = t.view(torch.bfloat16)
    return t


def _check_tensor(t, name, dtype, shape):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


class CommPlan:
    """A communication plan [MoonEPCommPlan]: device arrays owned by libmoonep."""

    def __init__(self, buffer: "Buffer", flags: int = 0):
        self._buffer = buffer
        self._st = MoonepCommPlan()
        check(_lib.load().moonep_plan_create(buffer._ctx, flags, ctypes.byref(self._st)),
              "moonep_plan_create")
        st = self._st
        R, E, B, K, S, NvS = st.R, st.E, st.B, st.K, st.S, st.NvS
        self.R, self.E, self.B, self.K, self.S, self.NvS, self.N = R, E, B, K, S, NvS, st.N
        self.flags = flags
        self.dst = _view(st.dst, (R, S * K), self)
        self.experts_to_copy = _view(st.experts_to_copy, (R, B), self)
        self.cu_seqlens = _view(st.cu_seqlens, (R, E + B), self)
        self.zero_fill_ranges = _view(st.zero_fill_ranges, (R, E + B, 2), self)
        self.remote_stats = _view(st.remote_stats, (R, 2), self)
        self.dup_counts = _view(st.dup_counts, (R, 2), self)
        if flags & _lib.PLAN_DUP_RECORDS:
            self.dup_groups = _view(st.dup_groups, (R, NvS, 3), self)
            self.dup_loffs = _view(st.dup_loffs, (R, NvS), self)
        else:
            self.dup_groups = self.dup_loffs = None

    @property
    def struct(self):
        return ctypes.byref(self._st)

    def clone(self) -> "CommPlan":
        """Deep copy of every array and scalar [MoonEPCommPlan.clone()]."""
        other = CommPlan(self._buffer, self.flags)
        check(_lib.load().moonep_plan_clone(self.struct, other.struct, _stream()),
              "moonep_plan_clone")
        return other

    def destroy(self):
        if getattr(self, "_st", None) is not None and self._st.internal:
            _lib.load().moonep_plan_destroy(ctypes.byref(self._st))

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


class Buffer:
    """Persistent resources of the balanced EP hot path [Buffer(...)].

    S tokens per rank, H hidden, K routes per token, E experts, R ranks
    (num_ep_ranks), B prefetch slots per rank (default E // R), token_padding
    rows of alignment per non-empty segment, num_sms SM cap (None: all)."""

    def __init__(self, S: int, H: int, K: int, E: int, num_ep_ranks: int, B: int | None = None,
                 token_padding: int = 128, num_sms: int | None = None,
                 zero_copy_views: bool = True, dup_records: bool = False):
        lib = _lib.load()
        R = num_ep_ranks
        B = E // R if B is None else B
        self.cfg = MoonepConfig(R=R, E=E, K=K, S=S, H=H, B=B, token_padding=token_padding,
                                num_sms=0 if num_sms is None else num_sms)
        self.R, self.E, self.K, self.S, self.H, self.B = R, E, K, S, H, B
        self.token_padding = token_padding
        nvs, nvsp = ctypes.c_int(), ctypes.c_int()
        check(lib.moonep_query_sizes(ctypes.byref(self.cfg), ctypes.byref(nvs),
                                     ctypes.byref(nvsp), None), "moonep_query_sizes")
        self.NvS, self.NvS_padded = nvs.value, nvsp.value
        torch.cuda.current_device()  # make sure the primary context exists
        h = ctypes.c_void_p()
        check(lib.moonep_ctx_create(ctypes.byref(self.cfg), int(zero_copy_views),
                                    ctypes.byref(h)), "moonep_ctx_create")
        self._ctx = h
        self._plan_flags = _lib.PLAN_DUP_RECORDS if dup_records else 0
        self._views = zero_copy_views

    # ----------------------------------------------------------- lifecycle
    @property
    def destroyed(self) -> bool:
        return self._ctx is None or bool(_lib.load().moonep_ctx_destroyed(self._ctx))

    def destroy(self) -> None:
        """Synchronise and release everything [Buffer.destroy()]; idempotent."""
        if self._ctx is not None:
            _lib.load().moonep_ctx_destroy(self._ctx)

    def __del__(self):
        try:
            if self._ctx is not None:
                _lib.load().moonep_ctx_free(self._ctx)
                self._ctx = None
        except Exception:
            pass

    @property
    def num_sms(self) -> int:
        return _lib.load().moonep_num_sms(self._ctx)

    # ------------------------------------------------------------- views
    def hidden_nvsh_buffer_view(self, rank: int | None = None) -> torch.Tensor:
        """Writable [NvS, H] bf16 window of rank `rank` (all ranks, [R*NvS, H],
        when rank is None) of the persistent hidden buffer."""
        lib = _lib.load()
        if rank is None:
            p = lib.moonep_hidden_view(self._ctx, 0)
            return _view(p, (self.R * self.NvS, self.H), self, torch.bfloat16)
        return _view(lib.moonep_hidden_view(self._ctx, rank), (self.NvS, self.H), self,
                     torch.bfloat16)

    def router_weight_buffer_view(self, rank: int | None = None) -> torch.Tensor:
        lib = _lib.load()
        if rank is None:
            return _view(lib.moonep_weight_view(self._ctx, 0), (self.R * self.NvS,), self,
                         torch.float32)
        return _view(lib.moonep_weight_view(self._ctx, rank), (self.NvS,), self, torch.float32)

    # -------------------------------------------------------------- plan
    def new_plan(self) -> CommPlan:
        return CommPlan(self, self._plan_flags)

    def plan(self, topk_experts_sk: torch.Tensor, tokens_per_expert: torch.Tensor | None = None,
             plan: CommPlan | None = None) -> CommPlan:
        """Run the online planner into `plan` (a new plan when None)."""
        R, S, K, E = self.R, self.S, self.K, self.E
        tk = _check_tensor(topk_experts_sk, "topk_experts_sk", torch.int32, (R, S, K))
        tp = None
        if tokens_per_expert is not None:
            tp = _check_tensor(tokens_per_expert, "tokens_per_expert", torch.int32, (R, E))
        plan = self.new_plan() if plan is None else plan
        check(_lib.load().moonep_plan(self._ctx, tk, tp, plan.struct, _stream()), "moonep_plan")
        return plan

    # ---------------------------------------------------------- dispatch
    def dispatch(self, hidden_sh: torch.Tensor, route_weights_sk: torch.Tensor | None = None,
                 topk_experts_sk: torch.Tensor | None = None,
                 tokens_per_expert: torch.Tensor | None = None, plan: CommPlan | None = None,
                 zero_copy: bool = False, router_weights_zero_copy: bool = False,
                 out: torch.Tensor | None = None, weights_out: torch.Tensor | None = None,
                 dedup: bool = False, plan_out: CommPlan | None = None):
        """Fresh dispatch (plan is None: plan then dispatch, into plan_out or
        a new plan) or plan-reuse dispatch [Buffer.dispatch].  dedup=True
        copies only the primary rows and expands the duplicates in an
        epilogue (same result; needs a Buffer made with dup_records=True).

        Returns (hidden_nvsh [R*NvS, H] bf16, route_weights_nvs [R*NvS] fp32 or
        None, cu_seqlens [R, E+B] int32 (None on plan reuse), plan)."""
        R, S, H, K, NvS = self.R, self.S, self.H, self.K, self.NvS
        hp = _check_tensor(hidden_sh, "hidden_sh", torch.bfloat16, (R, S, H))
        fresh = plan is None
        tk = tp = None
        if fresh:
            if topk_experts_sk is None:
                raise ValueError("a fresh dispatch needs topk_experts_sk")
            tk = _check_tensor(topk_experts_sk, "topk_experts_sk", torch.int32, (R, S, K))
            if tokens_per_expert is not None:
                tp = _check_tensor(tokens_per_expert, "tokens_per_expert", torch.int32,
                                   (R, self.E))
            plan = self.new_plan() if plan_out is None else plan_out
            check(_lib.load().moonep_plan(self._ctx, tk, tp, plan.struct, _stream()),
                  "moonep_plan")
        if out is None:
            out = self.hidden_nvsh_buffer_view() if zero_copy else torch.empty(
                (R * NvS, H), dtype=torch.bfloat16, device=hidden_sh.device)
        op = _check_tensor(out, "hidden_nvsh", torch.bfloat16, (R * NvS, H))
        wp = wop = None
        w_out = None
        if route_weights_sk is not None:
            wp = _check_tensor(route_weights_sk, "route_weights_sk", torch.float32, (R, S, K))
            if weights_out is None:
                weights_out = self.router_weight_buffer_view() if router_weights_zero_copy \
                    else torch.empty((R * NvS,), dtype=torch.float32, device=hidden_sh.device)
            wop = _check_tensor(weights_out, "route_weights_nvs", torch.float32, (R * NvS,))
            w_out = weights_out
        fn = "moonep_dispatch_dedup" if dedup else "moonep_dispatch"
        check(getattr(_lib.load(), fn)(self._ctx, plan.struct, hp, wp, op, wop, _stream()), fn)
        return out, w_out, (plan.cu_seqlens if fresh else None), plan

    # ----------------------------------------------------------- combine
    def combine(self, plan: CommPlan, hidden_nvsh: torch.Tensor,
                route_weights_nvs: torch.Tensor | None = None, out: torch.Tensor | None = None,
                weights_out: torch.Tensor | None = None, dedup: bool = False):
        """Gather and K-sum back to token-major [Buffer.combine].
        dedup=True first folds every rank's duplicate rows of a token into its
        primary row (fp32, one bf16 rounding, IN PLACE on hidden_nvsh), then
        sums the primaries only; needs a Buffer made with dup_records=True.
        Returns (hidden_sh [R, S, H] bf16, route_weights_sk [R, S, K] or None)."""
        R, S, H, K, NvS = self.R, self.S, self.H, self.K, self.NvS
        yp = _check_tensor(hidden_nvsh, "hidden_nvsh", torch.bfloat16, (R * NvS, H))
        if out is None:
            out = torch.empty((R, S, H), dtype=torch.bfloat16, device=hidden_nvsh.device)
        op = _check_tensor(out, "hidden_sh", torch.bfloat16, (R, S, H))
        wp = wop = None
        if route_weights_nvs is not None:
            wp = _check_tensor(route_weights_nvs, "route_weights_nvs", torch.float32, (R * NvS,))
            if weights_out is None:
                weights_out = torch.empty((R, S, K), dtype=torch.float32,
                                          device=hidden_nvsh.device)
            wop = _check_tensor(weights_out, "route_weights_sk", torch.float32, (R, S, K))
        else:
            weights_out = None
        fn = "moonep_combine_dedup" if dedup else "moonep_combine"
        check(getattr(_lib.load(), fn)(self._ctx, plan.struct, yp, wp, op, wop, _stream()), fn)
        return out, weights_out

    # --------------------------------------------------- weights / grads
    def prefetch_weight(self, plan: CommPlan, *weights: torch.Tensor, scales=None) -> None:
        """Fill the prefetch slots of every [E + R*B, ...] weight tensor given
        (gate, up, down, ...; at most 4) [Buffer.prefetch_weight].  bf16
        tensors [E + R*B, H, H'], or packed MXFP4 uint8 [E + R*B, H, H'/2]; with
        `scales`, the block-scale tensors [E + R*B, ...] of the same set, one
        per weight tensor (a complete set), all copied by one launch."""
        if not weights or len(weights) > 4:
            raise ValueError("prefetch_weight takes 1 to 4 weight tensors")
        rows = self.E + self.R * self.B
        if scales is None and all(w.dtype == torch.bfloat16 for w in weights):
            HHp = None
            ptrs = []
            for i, w in enumerate(weights):
                hh = w[0].numel() if w.dim() > 1 else 0
                HHp = hh if HHp is None else HHp
                if hh != HHp:
                    raise ValueError("all weight tensors must share H*H'")
                ptrs.append(_check_tensor(w, f"weight[{i}]", torch.bfloat16, (rows, *w.shape[1:])))
            check(_lib.load().moonep_prefetch_weight(self._ctx, plan.struct, len(ptrs),
                                                      _lib.ptr_array(ptrs), HHp, _stream()),
                  "moonep_prefetch_weight")
            return
        tensors = list(weights)
        if scales is not None:
            scales = list(scales)
            if len(scales) != len(weights):
                raise ValueError("scales must be a complete set: one per weight tensor")
            tensors += scales
        self.prefetch_rows(plan, tensors)

    def prefetch_rows(self, plan: CommPlan, tensors) -> None:
        """Fill the prefetch slots of up to 8 [E + R*B, ...] tensors of any
        dtype (rows copied byte for byte) in one launch [Buffer.prefetch_weight]."""
        tensors = list(tensors)
        if not tensors or len(tensors) > 8:
            raise ValueError("prefetch_rows takes 1 to 8 tensors")
        rows = self.E + self.R * self.B
        ptrs, rb = [], []
        for i, t in enumerate(tensors):
            _check_tensor(t, f"tensor[{i}]", t.dtype, (rows, *t.shape[1:]))
            ptrs.append(t.data_ptr())
            rb.append(t[0].numel() * t.element_size() if t.dim() > 1 else t.element_size())
        arr = (ctypes.c_int64 * len(rb))(*rb)
        check(_lib.load().moonep_prefetch_rows(self._ctx, plan.struct, len(ptrs),
                                                _lib.ptr_array(ptrs), arr, _stream()),
              "moonep_prefetch_rows")

    def prepare(self, hidden: torch.Tensor | None, topk: torch.Tensor,
                weights: torch.Tensor | None = None, num_tokens=None,
                tokens_per_expert: bool = True) -> torch.Tensor | None:
        """Pad this step's batch to the static capacity S and map invalid
        (negative) expert ids to expert 0 with zero weight, in place
        [vLLM MoonEPPrepareAndFinalize.prepare / _pad_to_capacity].  hidden
        [R, S, H] bf16 (or None), topk [R, S, K] int32, weights [R, S, K] fp32
        (or None): rank r's first num_tokens[r] rows hold its batch.  Returns
        tokens_per_expert [R, E] int32 of the prepared ids (or None)."""
        R, S, K, H = self.R, self.S, self.K, self.H
        hp = _check_tensor(hidden, "hidden", torch.bfloat16, (R, S, H)) if hidden is not None else None
        tp = _check_tensor(topk, "topk", torch.int32, (R, S, K))
        wp = _check_tensor(weights, "weights", torch.float32, (R, S, K)) if weights is not None else None
        nt = None
        if num_tokens is not None:
            vals = [int(v) for v in (num_tokens.tolist() if torch.is_tensor(num_tokens)
                                     else num_tokens)]
            if len(vals) != R:
                raise ValueError(f"num_tokens: expected {R} values")
            nt = (ctypes.c_int32 * R)(*vals)
        tpe = torch.empty((R, self.E), dtype=torch.int32, device="cuda") if tokens_per_expert else None
        check(_lib.load().moonep_prepare(self._ctx, nt, hp, tp, wp,
                                         tpe.data_ptr() if tpe is not None else None, _stream()),
              "moonep_prepare")
        return tpe

    def reduce_grad(self, plan: CommPlan, grads, reduce_buffers) -> None:
        """Add the slot gradients into their home experts and clear the used
        slots [Buffer.reduce_grad].  grads: [E, H, H'] fp32 tensors;
        reduce_buffers: matching [R, B, H, H'] fp32 tensors."""
        grads, reduce_buffers = list(grads), list(reduce_buffers)
        if not grads or len(grads) != len(reduce_buffers) or len(grads) > 4:
            raise ValueError("reduce_grad takes 1 to 4 (grad, reduce_buffer) pairs")
        HHp = grads[0][0].numel()
        gp, sp = [], []
        for i, (g, s) in enumerate(zip(grads, reduce_buffers)):
            gp.append(_check_tensor(g, f"grad[{i}]", torch.float32, (self.E, *g.shape[1:])))
            sp.append(_check_tensor(s, f"reduce_buffer[{i}]", torch.float32,
                                    (self.R, self.B, *g.shape[1:])))
            if g[0].numel() != HHp:
                raise ValueError("all gradients must share H*H'")
        check(_lib.load().moonep_reduce_redundant_grad(
            self._ctx, plan.struct, len(gp), _lib.ptr_array(gp), _lib.ptr_array(sp), HHp,
            _stream()), "moonep_reduce_redundant_grad")

    # ------------------------------------------------- rank-local forms
    # The per-rank shape of the path when each EP rank is its own GPU: one
    # exchange (the all-gather of every rank's [E] tokens_per_expert, see
    # gather_tokens_per_expert), then each rank plans its own routes and
    # moves its own tokens, with the other ranks' rows behind window pointers.
    def plan_rank(self, rank: int, topk_sk: torch.Tensor, hist_all: torch.Tensor,
                  plan: CommPlan | None = None) -> CommPlan:
        """Rank `rank`'s share of the plan [Buffer.dispatch planning, per
        rank]: topk_sk [S, K] int32 of that rank, hist_all [R, E] int32 the
        gathered per-rank histograms.  Writes the rank's dst row, the tables
        shared by every rank, and the rank's share of dup_counts."""
        tk = _check_tensor(topk_sk, "topk_sk", torch.int32, (self.S, self.K))
        hp = _check_tensor(hist_all, "hist_all", torch.int32, (self.R, self.E))
        plan = self.new_plan() if plan is None else plan
        check(_lib.load().moonep_plan_rank(self._ctx, int(rank), tk, hp, plan.struct, _stream()),
              "moonep_plan_rank")
        return plan

    def _windows(self, rows, weights, name):
        R, NvS, H = self.R, self.NvS, self.H
        if len(rows) != R:
            raise ValueError(f"{name}: expected {R} rank windows")
        rp = [_check_tensor(t, f"{name}[{j}]", torch.bfloat16, (NvS, H)) for j, t in enumerate(rows)]
        wp = None
        if weights is not None:
            if len(weights) != R:
                raise ValueError(f"{name}: expected {R} weight windows")
            wp = _lib.ptr_array([_check_tensor(t, f"{name} weights[{j}]", torch.float32, (NvS,))
                                 for j, t in enumerate(weights)])
        return _lib.ptr_array(rp), wp

    def dispatch_rank(self, plan: CommPlan, rank: int, hidden_sh: torch.Tensor,
                      route_weights_sk: torch.Tensor | None, windows, weight_windows=None):
        """Rank `rank`'s tokens into the R rank windows (each [NvS, H] bf16,
        its own tensor) and zero padding of the rank's own window
        [Buffer.dispatch, per rank]."""
        hp = _check_tensor(hidden_sh, "hidden_sh", torch.bfloat16, (self.S, self.H))
        wp = None
        if route_weights_sk is not None:
            wp = _check_tensor(route_weights_sk, "route_weights_sk", torch.float32,
                               (self.S, self.K))
        rows, wins = self._windows(windows, weight_windows, "windows")
        check(_lib.load().moonep_dispatch_rank(self._ctx, plan.struct, int(rank), hp, wp, rows,
                                               wins, _stream()), "moonep_dispatch_rank")

    def combine_rank(self, plan: CommPlan, rank: int, windows, weight_windows=None,
                     out: torch.Tensor | None = None):
        """Rank `rank`'s tokens gathered from the R rank windows and K-summed
        [Buffer.combine, per rank].  Returns (hidden_sh [S, H] bf16,
        route_weights_sk [S, K] fp32 or None)."""
        rows, wins = self._windows(windows, weight_windows, "windows")
        if out is None:
            out = torch.empty((self.S, self.H), dtype=torch.bfloat16, device="cuda")
        op = _check_tensor(out, "hidden_sh", torch.bfloat16, (self.S, self.H))
        w_out = None
        wop = None
        if weight_windows is not None:
            w_out = torch.empty((self.S, self.K), dtype=torch.float32, device="cuda")
            wop = w_out.data_ptr()
        check(_lib.load().moonep_combine_rank(self._ctx, plan.struct, int(rank), rows, wins, op,
                                              wop, _stream()), "moonep_combine_rank")
        return out, w_out

    # ------------------------------------------------------------ status
    def get_status(self) -> int:
        """Synchronise the current stream and return (and clear) the first
        error a kernel latched since the last call (0 when none)."""
        v = ctypes.c_int()
        check(_lib.load().moonep_get_status(self._ctx, ctypes.byref(v), _stream()),
              "moonep_get_status")
        return v.value


def gather_tokens_per_expert(tokens_per_expert: torch.Tensor, group=None) -> torch.Tensor:
    """The rank-local planner's one exchange step: every rank's [E] int32
    tokens_per_expert, all-gathered into [R, E] in rank order over
    torch.distributed (the group's ranks are the EP ranks).  Every rank then
    holds the same histogram, from which Buffer.plan_rank derives the same
    balance tables on every rank."""
    import torch.distributed as dist
    t = tokens_per_expert.to(torch.int32).contiguous()
    if t.dim() != 1:
        raise ValueError("tokens_per_expert: expected [E]")
    world = dist.get_world_size(group)
    parts = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(parts, t, group=group)
    return torch.stack(parts)


class BufferPool:
    """Decode-step Buffers at a few token capacities, made on first use.

    A Buffer's token capacity S is fixed at creation and every step pads its
    batch up to it, so a single buffer sized for the largest batch makes a
    small decode step pay for the largest one.  The pool maps a step's token
    count to a capacity by the vLLM integration's rule (MoonEPBufferPool: the
    smallest power of two that holds the tokens, kept within [min_tokens,
    max_tokens_per_rank]) and keeps one Buffer per capacity it has served, so
    the number of distinct buffers grows with log2(max / min) at most.  Every
    rank of a step must ask with the same token count, so that they agree on
    the capacity.  A count above max_tokens_per_rank is refused by get(): no
    buffer could hold that batch."""

    def __init__(self, max_tokens_per_rank: int, min_tokens: int = 1, **buffer_kwargs):
        if not 1 <= min_tokens <= max_tokens_per_rank:
            raise ValueError("need 1 <= min_tokens <= max_tokens_per_rank")
        if "S" in buffer_kwargs:
            raise ValueError("the pool chooses S; pass the other Buffer arguments only")
        self.max_tokens_per_rank = max_tokens_per_rank
        self.min_tokens = min_tokens
        self._buffer_kwargs = dict(buffer_kwargs)
        self._by_capacity: dict[int, Buffer] = {}

    def capacity_for(self, num_tokens: int) -> int:
        """The rule alone: smallest power of two >= num_tokens, clamped to
        [min_tokens, max_tokens_per_rank]."""
        p = 1
        while p < num_tokens:
            p <<= 1
        return min(max(p, self.min_tokens), self.max_tokens_per_rank)

    def get(self, num_tokens: int) -> tuple[int, Buffer]:
        """(capacity, Buffer of that capacity) for a step of num_tokens tokens
        per rank; the Buffer is created the first time its capacity is used."""
        if num_tokens < 0 or num_tokens > self.max_tokens_per_rank:
            raise ValueError(f"{num_tokens} tokens per rank: outside [0, "
                             f"{self.max_tokens_per_rank}]")
        cap = self.capacity_for(num_tokens)
        if cap not in self._by_capacity:
            self._by_capacity[cap] = Buffer(S=cap, **self._buffer_kwargs)
        return cap, self._by_capacity[cap]

    @property
    def capacities(self) -> list[int]:
        """Capacities that have a Buffer, ascending."""
        return sorted(self._by_capacity)

    def destroy(self) -> None:
        """Destroy every Buffer the pool made; the pool can be used again."""
        while self._by_capacity:
            _, buf = self._by_capacity.popitem()
            buf.destroy()
