"""Workload shapes of the structured-read denoise step.

Shapes only: no arithmetic of the method lives here.  The canvas length (256),
the 512-wide heads, the 26-label cap, the 0.1 entropy gate and the four noise
reads come from the DiffusionGemma pages (24-ai.news "How does diffusion text
generation differ?"; sotaaz.com "Getting it running on an A100" and "The server
accepts at most 26 alternatives per question"); GQA 8/2, d_model 2816, vocab
262144 and W=128 are the workload definitions the step is measured on.
"""
from dataclasses import dataclass, field
from typing import List, Tuple


@dataclass
class StepShape:
    name: str
    B: int                 # requests
    C: int                 # canvas tokens per request
    P: int                 # prompt (encoder KV) tokens per request (max when ragged)
    Hq: int
    Hkv: int
    d_head: int
    W: int                 # +-W canvas window
    D: int                 # d_model
    V: int                 # vocabulary
    slots: List[Tuple[int, int]] = field(default_factory=list)  # (canvas position, n_labels)
    R: int = 4             # reads per stage (samples)
    gate: float = 0.1      # slot entropy gate (nats)
    gamma: float = 0.0     # commit threshold (nats)
    all_open: bool = True  # every canvas position is a commit candidate
    steps: int = 1
    paged: bool = False
    page_size: int = 16


# Tiny correctness case: one request, one 4-label slot at canvas position 17.
TINY = StepShape("tiny_slot_read", B=1, C=32, P=64, Hq=2, Hkv=1, d_head=64, W=8,
                 D=128, V=1024, slots=[(17, 4)], gamma=3.2, all_open=True)

# Single structured read: 2-label yes/no, 26-label choice, 5-level score.
SINGLE_READ = StepShape("single_structured_read", B=1, C=256, P=2048, Hq=8, Hkv=2,
                        d_head=512, W=128, D=2816, V=262144,
                        slots=[(61, 2), (125, 26), (189, 5)], gamma=25.6,
                        all_open=False)

# Full-canvas denoise step with self-conditioning, 8 steps, threshold 0.1*256.
FULL_CANVAS = StepShape("full_canvas_step", B=1, C=256, P=4096, Hq=8, Hkv=2,
                        d_head=512, W=128, D=2816, V=262144,
                        slots=[(61, 2), (125, 26), (189, 5)], gamma=0.1 * 256,
                        all_open=True, steps=8)

# Mixed batched two-stage reads over a paged encoder KV (16-token pages).
MIXED_BATCH = StepShape("mixed_batched_reads", B=32, C=256, P=8192, Hq=8, Hkv=2,
                        d_head=512, W=128, D=2816, V=262144, gamma=25.6,
                        all_open=False, paged=True, page_size=16)

# Long context: one request with a 110,707-token prompt.
LONG_CONTEXT = StepShape("long_context_read", B=1, C=256, P=110707, Hq=8, Hkv=2,
                         d_head=512, W=128, D=2816, V=262144,
                         slots=[(61, 2), (125, 26), (189, 5)], gamma=25.6,
                         all_open=False)

ALL = {0: TINY, 1: SINGLE_READ, 2: FULL_CANVAS, 3: MIXED_BATCH, 4: LONG_CONTEXT}


def scaled(shape: StepShape, **kw) -> StepShape:
    """A copy of ``shape`` with some fields replaced (for reduced parity sizes)."""
    d = dict(shape.__dict__)
    d.update(kw)
    return StepShape(**d)
