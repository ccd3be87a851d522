"""ctypes declarations of the C ABI in include/moe_async.h (argument marshalling only)."""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_DEBUG_BOUNDS=1 selects the bounds-checked build of the same library
DEBUG_BOUNDS = os.environ.get("MOE_DEBUG_BOUNDS", "") == "1"
LIB_PATH = os.path.join(_HERE, "libmoe_async_debug.so" if DEBUG_BOUNDS else "libmoe_async.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_CAPACITY, MOE_ERR_DUPLICATE, MOE_ERR_STALE, \
    MOE_ERR_TIMEOUT, MOE_ERR_CUDA, MOE_ERR_UNSUPPORTED, MOE_ERR_BOUNDS = range(9)
MOE_F32, MOE_BF16 = 0, 1
MOE_POLICY_MTFS, MOE_POLICY_THRESHOLD, MOE_POLICY_RANKS = 0, 1, 2
MOE_EXPERT_SWIGLU, MOE_EXPERT_IDENTITY = 0, 1

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID", 2: "MOE_ERR_CAPACITY", 3: "MOE_ERR_DUPLICATE",
                4: "MOE_ERR_STALE", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_CUDA", 7: "MOE_ERR_UNSUPPORTED",
                8: "MOE_ERR_BOUNDS"}

# every symbol include/moe_async.h declares
EXPORTS = ("moe_async_create", "moe_async_route", "moe_async_enqueue", "moe_async_schedule_step", "moe_async_tick",
           "moe_async_schedule_steps", "moe_async_collect", "moe_async_wait", "moe_async_sync", "moe_async_get_stats",
           "moe_async_get_trace", "moe_async_snapshot", "moe_async_destroy",
           "moe_async_status_string", "moe_async_host_writable", "moe_async_profile", "moe_async_profile_read",
           "moe_async_stream_setup", "moe_async_stream_run", "moe_async_stream_trace", "moe_async_stream_stats",
           "moe_async_cancel", "moe_async_debug_append_record")

KERNEL_KINDS = ("enqueue", "schedule", "ffn1", "ffn2", "collect", "tick")


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "num_experts", "top_k", "hidden", "inter", "dtype", "has_shared",
        "max_slots", "bucket_capacity", "expert_kind", "trace_capacity")]


class Policy(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("kind", "max_groups", "min_batch", "fallback_groups")]


class Stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("pairs_executed", ctypes.c_int64),
                ("expert_runs", ctypes.c_int64), ("weight_bytes", ctypes.c_int64),
                ("tokens_combined", ctypes.c_int64), ("duplicates", ctypes.c_int64),
                ("stale", ctypes.c_int64), ("open_tokens", ctypes.c_int32),
                ("pending_pairs", ctypes.c_int32), ("ready", ctypes.c_int32),
                ("error", ctypes.c_int32), ("packed_weight_bytes", ctypes.c_int64),
                ("kernel_launches", ctypes.c_int64), ("cancelled", ctypes.c_int64)]


class StreamConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_requests", "max_steps", "stop_combines", "policy",
                                              "defrag_window", "history_window")] + \
               [("defrag_decay", ctypes.c_double)]


STREAM_POLICIES = {"mtfs": 0, "flfs": 1, "defrag": 2, "barrier": 3, "defrag_src": 4}


class StreamStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("ticks", "combined", "peak_transit", "peak_bucket", "num_queues")] + \
               [("peak_queue", ctypes.c_int32 * 16), ("occupancy_sum", ctypes.c_int64 * 16)]


class MoEError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


_lib = None


def load():
    """Load libmoe_async.so; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, U32P, I32P, F32P = ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    VPP = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "moe_async_create": [ctypes.POINTER(Config), VPP, VPP, VPP, VPP, VPP, VPP, P, ctypes.POINTER(P)],
        "moe_async_route": [F32P, I32, I32, I32, I32P, F32P, P],
        "moe_async_enqueue": [P, I32, I32, I32P, I32P, P, I32P, F32P, U32P, U32P, P],
        "moe_async_schedule_step": [P, I32, ctypes.POINTER(Policy), P],
        "moe_async_schedule_steps": [P, I32, ctypes.POINTER(Policy), I32, P],
        "moe_async_collect": [P, I32, I32, P, I32P, U32P, U32P, I32P, I32, P],
        "moe_async_tick": [P, I32, I32, I32P, I32P, P, I32P, F32P, U32P, U32P, ctypes.POINTER(Policy), I32, P, I32P,
                           U32P, U32P, I32P, I32, P],
        "moe_async_wait": [P, I32, ctypes.POINTER(Policy), I32, I32, P],
        "moe_async_sync": [P, P],
        "moe_async_get_stats": [P, P, ctypes.POINTER(Stats)],
        "moe_async_get_trace": [P, P, ctypes.POINTER(ctypes.c_int32), I32, ctypes.POINTER(ctypes.c_int32)],
        "moe_async_snapshot": [P, I32, P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                               I32, ctypes.POINTER(ctypes.c_int32)],
        "moe_async_destroy": [P, P],
        "moe_async_cancel": [P, I32, I32, I32P, P],
        "moe_async_debug_append_record": [P, I32, I32, I32, P],
        "moe_async_profile": [P, I32],
        "moe_async_profile_read": [P, P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64), I32],
        "moe_async_status_string": [ctypes.c_int],
        "moe_async_host_writable": [P, ctypes.c_int64],
        "moe_async_stream_setup": [P, ctypes.POINTER(StreamConfig), VPP, P, P, P, P, P, P, P],
        "moe_async_stream_stats": [P, P, ctypes.POINTER(StreamStats)],
        "moe_async_stream_run": [P, I32, I32, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32), P],
        "moe_async_stream_trace": [P, P, ctypes.POINTER(ctypes.c_int32), I32, ctypes.POINTER(ctypes.c_int32)],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_char_p if name == "moe_async_status_string" else ctypes.c_int
    _lib = lib
    return lib


def check(status, what):
    if status != MOE_OK:
        raise MoEError(status, what)
