"""CPU oracle for the Vegas hot path: TEST INFRASTRUCTURE, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.

Page cited throughout: "Resumo Técnico: Vegas – Decodificação Auto-Especulativa com
Atenção Esparsa Guiada por Verificação" (gist.science technical summary of paper
2602.07223), referred to as "Vegas §<section>".
"""
from .vegas import (  # noqa: F401
    widen_bf16,
    softmax_attention,
    verify_attention,
    verify_logits,
    aggregated_scores,
    aggregated_scores_grouped,
    select_topk,
    sparse_draft_attention,
    draft_step,
    iteration,
    selection_overlap,
    select_window,
    softmax,
    sample_inverse_cdf,
    argmax_lowest,
    accept_greedy,
    accept_sample,
    next_prefix_len,
    paged_slots,
)
