// Cost-model constants of pkv_policy_default. Written by serving_paged_gqa_gb300/calibrate.py (fit) from
// the calibration sweep; rebuild the library after changing them.
#pragma once
#define PKV_FIT_SOURCE "fitted on 1490 timed candidate plans, seeds [0, 1, 2, 3, 4]"
#define PKV_FIT_LAUNCH_US 7.93086
#define PKV_FIT_HBM_GBS 6108.02
#define PKV_FIT_CTA_GBS 24.2091
#define PKV_FIT_WQ_CTA_GBS 31.2778
#define PKV_FIT_TASK_US 0.05
#define PKV_FIT_TAIL 0.364288
#define PKV_FIT_MERGE_US 3.96352
#define PKV_FIT_MERGE_STATE_US 0.0145311
#define PKV_FIT_FUSED_US 0.794996
#define PKV_FIT_FUSED_STATE_US 0.108602
#define PKV_FIT_BUILD_US 4
